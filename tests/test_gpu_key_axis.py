"""The key-axis quality ablation through the kernels: the same seeded head as
tests/test_ablation_key_axis.py (T = 512 tokens, 4 query heads, outlier channels a*z + 5)
appended by the library's quantize-append kernels and attended by its decode kernel, for
the key schemes the library implements: per-channel keys (groups of 32 tokens), the same
with the 4 entries of each key row farthest from its median kept as binary16
(dense-and-sparse), and at 8 bits the symmetric per-token cache with and without those
entries. Each GPU output is first checked against the oracle's attention over the
oracle's state (parity, 2e-3); the error against unquantized binary16 keys and values is
then compared across schemes ("Sub-8-Bit KV Cache Quantization Is Not a Free Lever for an
RDNA4 Agent Swarm", § What the low-bit numbers actually cost).
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from kvq_testlib import ATOL  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from bit_kv_cache_09_gb300.cache import QuantizedKVCache  # noqa: E402

T, D, R, G, GV = 512, 128, 4, 32, 32


def _run(k16, v16, q16, *, bits, symmetric, k_out):
    cache = QuantizedKVCache(n_layers=1, batch=1, n_kv_heads=1, gqa_ratio=R, d_head=D, max_seq_len=T, bits=bits,
                             k_group=G, v_group=D if symmetric else GV, residual_len=0, symmetric=symmetric,
                             k_outliers=k_out)
    kd = torch.from_numpy(k16.reshape(1, T, 1, D)).cuda()
    vd = torch.from_numpy(v16.reshape(1, T, 1, D)).cuda()
    cache.append(0, 0, kd, vd)
    qd = torch.from_numpy(q16.reshape(1, R, D)).cuda()
    out = cache.attention(0, T, qd, 1.0 / np.sqrt(D)).cpu().numpy().reshape(R, D)
    cache.check_errors()
    if symmetric:
        st = oracle.cache_state_sym(k16, v16, d=D, k_outliers=k_out)
        kq, vq = oracle.dequantize_state_sym(st, d=D)
    else:
        st = oracle.cache_state(k16, v16, d=D, bits=bits, G=G, Gv=GV, R=0, k_outliers=k_out)
        kq, vq = oracle.dequantize_state(st, d=D, bits=bits, G=G, Gv=GV, R=0)
    ref_q = oracle.attention(q16, kq, vq, 1.0 / np.sqrt(D))
    assert float(np.abs(out - ref_q).max()) <= ATOL  # the kernels compute the oracle's attention
    return out


@pytest.fixture(scope="module")
def errors():
    res = {}
    for n_out, gain in ((4, 20.0), (6, 50.0)):
        k16 = synth.gen_k(77, 0, [0], range(T), 1, D, n_out, gain)[0, :, 0]
        v16 = synth.gen_v(77, 0, [0], range(T), 1, D)[0, :, 0]
        q16 = synth.gen_q(77, 0, [0], T, R, D)[0]
        ref = oracle.attention(q16, k16.astype(np.float32), v16.astype(np.float32), 1.0 / np.sqrt(D))
        for bits in (8, 4, 2):
            for k_out in (0, 4):
                out = _run(k16, v16, q16, bits=bits, symmetric=0, k_out=k_out)
                res[(n_out, gain, bits, "per-channel", k_out)] = float(np.abs(out - ref).max())
        for k_out in (0, 4):
            out = _run(k16, v16, q16, bits=8, symmetric=1, k_out=k_out)
            res[(n_out, gain, 8, "per-token-sym", k_out)] = float(np.abs(out - ref).max())
    print("\noutliers  bits  scheme           | max-abs error, no entries / 4 isolated entries per key row")
    for n_out, gain in ((4, 20.0), (6, 50.0)):
        for bits, scheme in ((8, "per-channel"), (8, "per-token-sym"), (4, "per-channel"), (2, "per-channel")):
            print(f"{n_out} x {gain:4.0f}  int{bits}  {scheme:16s} | {res[(n_out, gain, bits, scheme, 0)]:.2e} / "
                  f"{res[(n_out, gain, bits, scheme, 4)]:.2e}")
    return res


def test_isolated_entries_cut_the_error(errors):
    for n_out, gain in ((4, 20.0), (6, 50.0)):
        for bits in (4, 2):
            assert errors[(n_out, gain, bits, "per-channel", 4)] < errors[(n_out, gain, bits, "per-channel", 0)]
        assert errors[(n_out, gain, 8, "per-token-sym", 4)] < errors[(n_out, gain, 8, "per-token-sym", 0)]


def test_per_channel_int8_beats_per_token_int8(errors):
    # one scale per token is set by the token's outlier channels; per-channel groups are not
    for n_out, gain in ((4, 20.0), (6, 50.0)):
        assert errors[(n_out, gain, 8, "per-channel", 0)] < errors[(n_out, gain, 8, "per-token-sym", 0)]


def test_error_grows_as_bits_drop(errors):
    for n_out, gain in ((4, 20.0), (6, 50.0)):
        for k_out in (0, 4):
            e = [errors[(n_out, gain, b, "per-channel", k_out)] for b in (8, 4, 2)]
            assert e[0] < e[1] < e[2]
