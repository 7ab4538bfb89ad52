"""Quality ablation on synthetic data: keys quantized per channel (groups of G tokens,
the kernels' scheme) versus per token (groups of Gv channels, the values' scheme), and
per channel with the 4 entries of each key row farthest from its median kept aside as
binary16 (dense-and-sparse), at 8, 4 and 2 bits, measured as the decode-attention output
error and the KL divergence of the attention probabilities against unquantized binary16
keys and values.

The pages argue that keys carry outlier channels, so per-channel key grouping keeps
low-bit attention usable where per-token grouping breaks ("KV Cache Quantization —
8-bit and 4-bit", § The outlier problem: keys have outlier channels; "Sub-8-Bit KV
Cache Quantization Is Not a Free Lever for an RDNA4 Agent Swarm", § The cache is two
distributions, not one; § What the low-bit numbers actually cost, on per-vector
dense-and-sparse outlier isolation). Everything here runs on the oracle's quantizer and its
binary64 attention; the table is printed (pytest -s) and a few robust orderings are
asserted. The generator's outlier channels are a*z + 5 (z standard normal), i.e.
large in magnitude and in spread across tokens.
"""

import numpy as np
import pytest

import oracle
import synth

T, D, R = 512, 128, 4
G, GV = 32, 32


def _f16(pattern: int) -> np.float32:
    return np.array([pattern], np.uint16).view(np.float16).astype(np.float32)[0]


def _per_token_keys(k16, bits):
    """Keys quantized per token over groups of GV channels with the oracle's quantizer."""
    out = np.zeros(k16.shape, np.float32)
    qmin = np.float32(-(1 << (bits - 1)))
    for t in range(k16.shape[0]):
        for j in range(0, k16.shape[1], GV):
            g = k16[t, j:j + GV]
            s, z = oracle.quant_params(g, bits)
            u = oracle.quantize_values(g, bits, s, z)
            out[t, j:j + GV] = _f16(s) * ((u.astype(np.float32) + qmin) - _f16(z))
    return out


def _probs(q, k, scale):
    sc = (q.astype(np.float64) @ k.astype(np.float64).T) * scale
    sc -= sc.max(axis=1, keepdims=True)
    p = np.exp(sc)
    return p / p.sum(axis=1, keepdims=True)


def _kl(p, q):
    return float(np.mean(np.sum(p * (np.log(p) - np.log(q)), axis=1)))


def ablation(n_out, gain, bits, seed=77):
    k16 = synth.gen_k(seed, 0, [0], range(T), 1, D, n_out, gain)[0, :, 0]
    v16 = synth.gen_v(seed, 0, [0], range(T), 1, D)[0, :, 0]
    q16 = synth.gen_q(seed, 0, [0], T, R, D)[0]
    scale = 1.0 / np.sqrt(D)
    st = oracle.cache_state(k16, v16, d=D, bits=bits, G=G, Gv=GV, R=0)
    k_ch, v_hat = oracle.dequantize_state(st, d=D, bits=bits, G=G, Gv=GV, R=0)
    k_tok = _per_token_keys(k16, bits)
    kf, vf = k16.astype(np.float32), v16.astype(np.float32)
    ref = oracle.attention(q16, kf, vf, scale)
    p_ref = _probs(q16, kf, scale)
    st_o = oracle.cache_state(k16, v16, d=D, bits=bits, G=G, Gv=GV, R=0, k_outliers=4)
    k_cho, _ = oracle.dequantize_state(st_o, d=D, bits=bits, G=G, Gv=GV, R=0)
    res = {}
    for name, kq in (("per-channel", k_ch), ("per-token", k_tok), ("per-channel+4", k_cho)):
        out = oracle.attention(q16, kq, v_hat, scale)
        res[name] = (float(np.abs(out - ref).max()), _kl(p_ref, _probs(q16, kq, scale)))
    return res


CASES = [(4, 20.0, b) for b in (8, 4, 2)] + [(6, 50.0, b) for b in (8, 4, 2)]


@pytest.fixture(scope="module")
def table():
    rows = {c: ablation(*c) for c in CASES}
    print("\noutliers  bits | out err per-channel  per-token  per-channel+4 | KL per-channel  per-token  per-channel+4")
    for (n_out, gain, bits), r in rows.items():
        print(f"{n_out} x {gain:4.0f}  int{bits} | {r['per-channel'][0]:.2e}  {r['per-token'][0]:.2e}  "
              f"{r['per-channel+4'][0]:.2e} | {r['per-channel'][1]:.2e}  {r['per-token'][1]:.2e}  {r['per-channel+4'][1]:.2e}")
    return rows


def test_eight_bit_is_close_for_both_axes(table):
    for (n_out, gain, bits), r in table.items():
        if bits == 8:
            assert r["per-channel"][1] < 1e-2 and r["per-token"][1] < 1e-2


def test_per_channel_keys_win_with_moderate_outliers(table):
    # the kernels' scheme: per-channel keys beat per-token keys at 8 and 4 bits
    for bits in (8, 4):
        r = table[(4, 20.0, bits)]
        assert r["per-channel"][1] < r["per-token"][1]
        assert r["per-channel"][0] < r["per-token"][0]


def test_error_grows_as_bits_drop(table):
    for n_out, gain in ((4, 20.0), (6, 50.0)):
        for axis in ("per-channel", "per-token"):
            kls = [table[(n_out, gain, b)][axis][1] for b in (8, 4, 2)]
            assert kls[0] < kls[1] < kls[2]


def test_isolated_entries_cut_the_error_of_per_channel_keys(table):
    # four isolated entries per key row take the outlier channels' extremes out of the
    # per-channel groups: the attention KL drops at every width for both outlier models
    for (n_out, gain, bits), r in table.items():
        assert r["per-channel+4"][1] < r["per-channel"][1] / 3, (n_out, gain, bits)
        if bits < 8:
            assert r["per-channel+4"][0] < r["per-channel"][0]
