"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print, a hand-derived worked example (tests/golden/), a library routine
(numpy's binary16 conversion, torch's float64 attention), a closed form, an
invariant, or the pages' error bound.
"""

import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _f16(x):
    return np.asarray(x, np.float16)


def _bits(x):
    return _f16(x).view(np.uint16)


# ----------------------------------------------------------------------------- binary16 conversions
def test_f16_widening_matches_numpy_for_every_pattern():
    pats = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = pats.view(np.float16).astype(np.float32)
    got = np.array([oracle.f32_from_f16(int(p)) for p in pats], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _conversion_probe_values():
    rng = np.random.default_rng(1)
    vals = [rng.standard_normal(4000).astype(np.float32) * s for s in (1e-6, 1e-3, 1.0, 100.0, 3e4)]
    # exact midpoints between neighbouring binary16 values (ties), and points just beside them
    h = rng.integers(0, 0x7BFF, 4000).astype(np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    mid = ((lo + hi) / 2).astype(np.float32)  # exact in binary32
    vals += [mid, np.nextafter(mid, np.float32(np.inf)), np.nextafter(mid, np.float32(-np.inf))]
    vals.append(np.array([65504, 65505, 65519, 65520, 65536, 1e9, 2.0**-24, 2.0**-25, 2.0**-26, 3 * 2.0**-26,
                          0.0, 6.1e-5, 6.0e-5], np.float32))
    v = np.concatenate(vals).astype(np.float32)
    return np.concatenate([v, -v])


def test_f16_round_nearest_even_matches_numpy():
    x = _conversion_probe_values()
    ref = x.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f16_from_f32_rne(float(v)) for v in x], np.uint16)
    assert np.array_equal(got, ref)


def test_f16_round_up_is_the_binary16_ceiling():
    x = _conversion_probe_values()
    x = x[np.abs(x) <= 65504]
    for v in x:
        h = np.uint16(oracle.f16_from_f32_ru(float(v)))
        hv = np.float64(h.view(np.float16))
        assert hv >= float(v)
        below = np.float64(np.nextafter(h.view(np.float16), np.float16(-np.inf)))
        assert below < float(v)


# ----------------------------------------------------------------------------- quantizer pins
def test_worked_example_minus_0p1_to_3p0():
    g = json.load(open(os.path.join(GOLDEN, "quant_worked_example.json")))
    x = _f16(g["inputs"])
    for c in g["cases"]:
        s, z = oracle.quant_params(x, c["bits"])
        assert s == int(c["scale_f16"], 16)
        assert z == int(c["zp_f16"], 16)
        u = oracle.quantize_values(x, c["bits"], s, z)
        assert u.tolist() == c["u"]


def test_round_half_to_even_ties():
    g = json.load(open(os.path.join(GOLDEN, "quant_ties.json")))
    for c in g["cases"]:
        x = _f16(c["x"])
        s, z = oracle.quant_params(x, c["bits"])
        assert (s, z) == (int(c["scale_f16"], 16), int(c["zp_f16"], 16))
        assert oracle.quantize_values(x, c["bits"], s, z).tolist() == c["u"]


def test_int_ranges():
    # int8 [-128, 127] and int4 [-8, 7] as printed; int2 read as [-2, 1]
    assert (oracle.qmin(8), oracle.qmax(8)) == (-128, 127)
    assert (oracle.qmin(4), oracle.qmax(4)) == (-8, 7)
    assert (oracle.qmin(2), oracle.qmax(2)) == (-2, 1)


def test_identity_case_int8():
    x = _f16(np.arange(-128, 128))
    np.random.default_rng(0).shuffle(x)
    s, z = oracle.quant_params(x, 8)
    assert np.uint16(s).view(np.float16) == 1.0
    assert np.uint16(z).view(np.float16) == 0.0
    u = oracle.quantize_values(x, 8, s, z)
    assert np.array_equal(u.astype(np.int32) - 128, x.astype(np.int32))


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_on_grid_round_trip_is_exact(bits):
    rng = np.random.default_rng(bits)
    qmin, qmax = oracle.qmin(bits), oracle.qmax(bits)
    for trial in range(200):
        s = 2.0 ** int(rng.integers(-8, 4))
        zp = int(rng.integers(-40, 41))
        n = int(rng.integers(2, 130))
        q = rng.integers(qmin, qmax + 1, n)
        q[0], q[-1] = qmin, qmax
        x = (s * (q - zp)).astype(np.float64)
        xh = _f16(x)
        assert np.array_equal(xh.astype(np.float64), x)  # on the binary16 grid
        sh, zh = oracle.quant_params(xh, bits)
        assert np.uint16(sh).view(np.float16) == s
        assert np.uint16(zh).view(np.float16) == zp
        u = oracle.quantize_values(xh, bits, sh, zh)
        assert np.array_equal(u.astype(np.int64), q - qmin)
        back = np.array([oracle.dequantize_value(int(v), bits, sh, zh) for v in u], np.float32)
        assert np.array_equal(back.view(np.uint32), x.astype(np.float32).view(np.uint32))


def _groups(rng, n_groups, size):
    out = []
    for i in range(n_groups):
        kind = i % 5
        if kind == 0:
            x = rng.standard_normal(size)
        elif kind == 1:
            x = rng.uniform(-0.1, 3.0, size)  # lopsided, as in the pages' example
        elif kind == 2:
            x = rng.standard_normal(size) * 20 + 5  # an outlier channel
        elif kind == 3:
            x = rng.standard_normal(size) * 1e-3 + 7.0  # far from zero, narrow
        else:
            x = rng.standard_normal(size) * 300.0
        out.append(_f16(x))
    return out


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_error_bound_half_step(bits):
    """|x - x_hat| <= scale/2 ("KV Cache Quantization — 8-bit and 4-bit", § Integer quantization in one screen)."""
    rng = np.random.default_rng(100 + bits)
    qmin, qmax = oracle.qmin(bits), oracle.qmax(bits)
    for x in _groups(rng, 300, 32) + _groups(rng, 50, 128):
        sh, zh = oracle.quant_params(x, bits)
        s = float(np.uint16(sh).view(np.float16))
        u = oracle.quantize_values(x, bits, sh, zh)
        assert u.max() <= qmax - qmin
        xd = x.astype(np.float64)
        xhat = np.array([oracle.dequantize_value(int(v), bits, sh, zh) for v in u], np.float64)
        err = np.abs(xd - xhat)
        zp = float(np.uint16(zh).view(np.float16))
        assert abs(zp) <= 2048 and zp == int(zp)  # an exact binary16 integer
        if xd.max() > xd.min():  # (a constant group is widened to include 0)
            assert u[int(np.argmin(xd))] == 0  # the smallest value lands on q_min
        assert err.max() <= s / 2 * (1 + 2.0**-20) + 1e-30, (bits, err.max(), s)


def test_narrow_groups_far_from_zero_keep_the_half_step_bound(golden_dir):
    """Hand-derived groups whose zero point would exceed the binary16 integers under the
    range rule alone: the widened scale max|x| / (2048 - 2^bits) (tests/golden/
    quant_far_from_zero.json) keeps the zero point exact and |x - x_hat| <= scale/2."""
    g = json.load(open(os.path.join(golden_dir, "quant_far_from_zero.json")))
    for case in g["cases"]:
        bits = case["bits"]
        x = _f16(case["x"])
        sh, zh = oracle.quant_params(x, bits)
        assert sh == int(case["scale_f16"], 16) and zh == int(case["zp_f16"], 16), (bits, hex(sh), hex(zh))
        u = oracle.quantize_values(x, bits, sh, zh)
        assert u.tolist() == case["u"]
        s = float(np.uint16(sh).view(np.float16))
        for xi, ui in zip(x.astype(np.float64), u):
            assert abs(oracle.dequantize_value(int(ui), bits, sh, zh) - xi) <= s / 2


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_near_constant_groups_anywhere_keep_the_half_step_bound(bits):
    """Groups of two or three neighbouring binary16 values at every magnitude from 2^-10
    to 60000, both signs: the stored zero point is an exact integer and every value is
    within half a (stored) step of its reconstruction."""
    for e in range(-10, 16):
        for sign in (1.0, -1.0):
            c = np.float16(sign * 1.37 * 2.0**e)
            up = np.nextafter(c, np.float16(np.inf))
            dn = np.nextafter(c, np.float16(-np.inf))
            for grp in ([c, up], [dn, c, up], [c, c, up, c]):
                x = _f16(grp)
                if not np.isfinite(x.astype(np.float64)).all():
                    continue
                sh, zh = oracle.quant_params(x, bits)
                s = float(np.uint16(sh).view(np.float16))
                zp = float(np.uint16(zh).view(np.float16))
                assert abs(zp) <= 2048 and zp == int(zp)
                u = oracle.quantize_values(x, bits, sh, zh)
                for xi, ui in zip(x.astype(np.float64), u):
                    assert abs(oracle.dequantize_value(int(ui), bits, sh, zh) - xi) <= s / 2 * (1 + 2.0**-20)


@pytest.mark.parametrize("bits", [2, 4, 8])
def test_scale_is_range_over_levels_rounded_up(bits):
    """scale = (x_max - x_min)/(q_max - q_min), stored in binary16 rounded up; a narrow
    group far from zero takes max|x| / (2048 - 2^bits) when that is larger."""
    rng = np.random.default_rng(200 + bits)
    N = oracle.qmax(bits) - oracle.qmin(bits)
    widened = 0
    for x in _groups(rng, 200, 64):
        xd = x.astype(np.float64)
        if xd.max() == xd.min():
            continue  # constant groups follow the widening rule (test_degenerate_groups)
        far = np.abs(xd).max() / (2048 - 2**bits)
        exact = max((xd.max() - xd.min()) / N, far)
        widened += far > (xd.max() - xd.min()) / N
        sh, _ = oracle.quant_params(x, bits)
        s = np.uint16(sh).view(np.float16)
        below = np.float64(np.nextafter(s, np.float16(-np.inf)))
        # rounded up from a binary32 quotient: within one binary16 step above, never a step below
        assert float(s) >= exact * (1 - 2.0**-22)
        assert below < exact * (1 + 2.0**-22)
    assert widened > 0  # the narrow groups around 7.0 take the wider scale


def test_degenerate_groups():
    for bits in (2, 4, 8):
        z = _f16(np.zeros(16))
        sh, zh = oracle.quant_params(z, bits)
        assert sh == 0x3C00
        u = oracle.quantize_values(z, bits, sh, zh)
        assert all(oracle.dequantize_value(int(v), bits, sh, zh) == 0.0 for v in u)
        for c in (2.0, -3.5, 1e-3, 60000.0):
            x = _f16(np.full(8, c))
            sh, zh = oracle.quant_params(x, bits)
            s = float(np.uint16(sh).view(np.float16))
            u = oracle.quantize_values(x, bits, sh, zh)
            xhat = oracle.dequantize_value(int(u[0]), bits, sh, zh)
            assert abs(xhat - float(x[0])) <= s / 2 * (1 + 2.0**-20)


# ----------------------------------------------------------------------------- bytes accounting
def test_bytes_formula_worked_example():
    g = json.load(open(os.path.join(GOLDEN, "kv_bytes_examples.json")))["worked_example"]
    L, H, d, S = g["L"], g["n_kv"], g["d_head"], g["S"]
    assert oracle.kv_bytes(L, H, d, 1, 16) == g["fp16_bytes_per_token"]
    assert oracle.kv_bytes(L, H, d, 1, 8) == g["elements_per_token"]  # one byte per element
    assert round(oracle.kv_bytes(L, H, d, S, 16) / 1e9, 1) == g["gb_fp16_approx"]
    assert round(oracle.kv_bytes(L, H, d, S, 8) / 1e9, 1) == g["gb_int8_approx"]
    assert round(oracle.kv_bytes(L, H, d, S, 4) / 1e9, 1) == g["gb_int4_approx"]


def test_bytes_per_token_table():
    g = json.load(open(os.path.join(GOLDEN, "kv_bytes_examples.json")))["per_token_table"]
    # the model's (L, n_kv, d) product is fixed by the fp16 row: 160 KiB = 2 * 2 B * L*n_kv*d
    prod = g["fp16_kib_per_token"] * 1024 // 4
    for row in g["rows"]:
        per_tok = oracle.kv_bytes(1, 1, prod, 1, row["bits"])
        assert per_tok == row["kib_per_token"] * 1024
        turn = oracle.kv_bytes(1, 1, prod, g["turn_tokens"], row["bits"]) / 2**30
        assert round(turn, 2) == row["gib_per_turn"]


def test_block_scale_overhead_64k():
    g = json.load(open(os.path.join(GOLDEN, "kv_bytes_examples.json")))["block_scale_64k"]
    prod = g["fp16_kib_per_token"] * 1024 // 4
    T = g["tokens"]
    assert oracle.kv_bytes(1, 1, prod, T, 16) / 2**30 == g["fp16_gib"]
    kib8 = oracle.kv_bytes(1, 1, prod, 1, 8, g["meta_bytes"], g["group_elems"]) / 1024
    lo, hi = g["int8_kib_per_token_range"]
    assert lo <= kib8 <= hi and kib8 == hi
    assert round(oracle.kv_bytes(1, 1, prod, T, 8, g["meta_bytes"], g["group_elems"]) / 2**30) == g["int8_gib_approx"]
    kib4 = oracle.kv_bytes(1, 1, prod, 1, 4, g["meta_bytes"], g["group_elems"]) / 1024
    assert kib4 == g["int4_kib_per_token"]
    gib4 = oracle.kv_bytes(1, 1, prod, T, 4, g["meta_bytes"], g["group_elems"]) / 2**30
    assert gib4 == 1.125 and abs(gib4 - g["int4_gib_approx"]) <= 0.005  # printed to two places


# ----------------------------------------------------------------------------- attention pins
def _sdpa64(q, k, v, scale):
    q = torch.as_tensor(np.asarray(q, np.float64))[None, :, None, :]  # [1, r, 1, d]
    k = torch.as_tensor(np.asarray(k, np.float64))[None, None].expand(1, q.shape[1], -1, -1)
    v = torch.as_tensor(np.asarray(v, np.float64))[None, None].expand(1, q.shape[1], -1, -1)
    o = torch.nn.functional.scaled_dot_product_attention(q, k, v, scale=scale)
    return o[0, :, 0, :].numpy()


@pytest.mark.parametrize("T,d,r", [(1, 8, 1), (5, 8, 2), (37, 16, 4), (300, 128, 8)])
def test_attention_matches_torch_float64(T, d, r):
    rng = np.random.default_rng(T * 7 + d)
    q = _f16(rng.standard_normal((r, d)))
    k = rng.standard_normal((T, d)).astype(np.float32) * 3
    v = rng.standard_normal((T, d)).astype(np.float32)
    scale = 1 / math.sqrt(d)
    got = oracle.attention(q, k, v, scale)
    ref = _sdpa64(q.astype(np.float64), k, v, scale)
    assert np.abs(got - ref).max() < 1e-6


def test_attention_invariants():
    rng = np.random.default_rng(5)
    T, d = 64, 16
    k = rng.standard_normal((T, d)).astype(np.float32)
    v = rng.standard_normal((T, d)).astype(np.float32)
    # zero query: uniform weights -> the mean of the values
    o = oracle.attention(np.zeros((1, d), np.float16), k, v, 0.25)
    assert np.abs(o[0] - v.astype(np.float64).mean(0)).max() < 1e-6
    # one dominant score -> that token's value
    kk = np.zeros((T, d), np.float32)
    kk[17, 0] = 100.0
    q = np.zeros((1, d), np.float16)
    q[0, 0] = 1.0
    o = oracle.attention(q, kk, v, 1.0)
    assert np.abs(o[0] - v[17]).max() < 1e-6


@pytest.mark.parametrize("bits,G,Gv,R", [(8, 32, 128, 0), (4, 128, 64, 128), (2, 32, 32, 128)])
def test_on_grid_cache_attention_equals_textbook(bits, G, Gv, R):
    """Keys and values on each group's grid quantize exactly, so attention over the
    quantized cache equals torch's float64 attention over the raw binary16 inputs."""
    rng = np.random.default_rng(bits)
    d, T, r = 128, 300, 4
    qmin, qmax = oracle.qmin(bits), oracle.qmax(bits)
    R_eff = R if R > 0 else G
    Tq = (T // R_eff) * R_eff
    k = np.zeros((T, d))
    for g in range(T // G):
        for c in range(d):
            s = 2.0 ** int(rng.integers(-6, 0))
            zp = int(rng.integers(-3, 4))
            qs = rng.integers(qmin, qmax + 1, G)
            qs[0], qs[-1] = qmin, qmax
            k[g * G:(g + 1) * G, c] = s * (qs - zp)
    k[(T // G) * G:] = rng.standard_normal((T - (T // G) * G, d))
    v = np.zeros((T, d))
    for t in range(T):
        for j in range(d // Gv):
            s = 2.0 ** int(rng.integers(-6, 0))
            zp = int(rng.integers(-3, 4))
            qs = rng.integers(qmin, qmax + 1, Gv)
            qs[0], qs[-1] = qmin, qmax
            v[t, j * Gv:(j + 1) * Gv] = s * (qs - zp)
    k16, v16 = _f16(k), _f16(v)
    assert np.array_equal(k16[:Tq].astype(np.float64), k[:Tq])
    st = oracle.cache_state(k16, v16, d=d, bits=bits, G=G, Gv=Gv, R=R)
    kh, vh = oracle.dequantize_state(st, d=d, bits=bits, G=G, Gv=Gv, R=R)
    assert np.array_equal(kh, k16.astype(np.float32))
    assert np.array_equal(vh, v16.astype(np.float32))
    q = _f16(rng.standard_normal((r, d)))
    got = oracle.attention(q, kh, vh, 1 / math.sqrt(d))
    ref = _sdpa64(q.astype(np.float64), k16.astype(np.float64), v16.astype(np.float64), 1 / math.sqrt(d))
    assert np.abs(got - ref).max() < 1e-6


# ----------------------------------------------------------------------------- quantization axes
def test_keys_per_channel_values_per_token():
    """Keys are grouped along tokens per channel, values along channels per token
    ("Sub-8-Bit KV Cache Quantization Is Not a Free Lever for an RDNA4 Agent Swarm",
    § The cache is two distributions, not one). A huge key channel and a huge value
    token must not spoil the other channels / tokens."""
    rng = np.random.default_rng(9)
    d, T, G, Gv, bits = 128, 64, 32, 128, 8
    k = rng.standard_normal((T, d))
    k[:, 5] *= 1000.0  # outlier key channel
    v = rng.standard_normal((T, d)) * 0.5
    v[7, :] *= 1000.0  # outlier value token
    k16, v16 = _f16(k), _f16(v)
    st = oracle.cache_state(k16, v16, d=d, bits=bits, G=G, Gv=Gv, R=0)
    kh, vh = oracle.dequantize_state(st, d=d, bits=bits, G=G, Gv=Gv, R=0)
    ek = np.abs(kh - k16.astype(np.float32))
    ev = np.abs(vh - v16.astype(np.float32))
    assert np.delete(ek, 5, axis=1).max() < 0.02  # ordinary channels keep a fine step
    assert ek[:, 5].max() > 0.5  # the outlier channel has its own coarse one
    assert np.delete(ev, 7, axis=0).max() < 0.01
    assert ev[7].max() > 0.5
    # every key group's metadata is per channel: G tokens share one (scale, zp) per channel
    assert st.k_meta.shape == (T // G, d, 2)
    assert st.v_meta.shape == ((T + 1) // 2, d // Gv, 4)  # pair records
    assert oracle.value_meta(st).shape == (T, d // Gv, 2)


def test_residual_window_keeps_newest_tokens_in_f16():
    rng = np.random.default_rng(11)
    d, T, G, Gv, R, bits = 128, 300, 32, 64, 128, 4
    k16 = _f16(rng.standard_normal((T, d)))
    v16 = _f16(rng.standard_normal((T, d)))
    st = oracle.cache_state(k16, v16, d=d, bits=bits, G=G, Gv=Gv, R=R)
    assert st.Tq == 256 and st.k_codes.shape[0] == 256
    for t in range(256, T):
        assert np.array_equal(st.k_resid[t % R], k16[t].view(np.uint16))
    kh, _ = oracle.dequantize_state(st, d=d, bits=bits, G=G, Gv=Gv, R=R)
    assert np.array_equal(kh[256:], k16[256:].astype(np.float32))
    # R = 0: the residual holds T mod G tokens
    st0 = oracle.cache_state(k16, v16, d=d, bits=bits, G=G, Gv=Gv, R=0)
    assert st0.Tq == (T // G) * G


# ----------------------------------------------------------------------------- packed layout against its written rules
def _golden_layout(golden_dir):
    return json.load(open(os.path.join(golden_dir, "layout_bytes.json")))


def test_key_rows_match_hand_derived_bytes(golden_dir):
    """Key rows packed by the oracle against bytes derived by hand from the layout text
    (tests/golden/layout_bytes.json): bit order inside a byte, byte order, code width."""
    d = 128
    for case in _golden_layout(golden_dir)["k_rows"]:
        bits = case["bits"]
        nbytes = d * bits // 8
        if "pattern" in case:
            c = np.arange(d)
            u = {"c": c, "c % 16": c % 16, "(c + c // 4) % 4": (c + c // 4) % 4}[case["pattern"]].astype(np.uint8)
            if case.get("bytes_hex") == "range":
                want = np.arange(nbytes, dtype=np.uint8)
            else:
                per = [int(x, 16) for x in case["period"]]
                want = np.array([per[k % len(per)] for k in range(nbytes)], np.uint8)
        else:
            u = np.zeros(d, np.uint8)
            for ch, code in case["codes"].items():
                u[int(ch)] = code
            want = np.zeros(nbytes, np.uint8)
            for k, v in case["nonzero"].items():
                want[int(k)] = int(v, 16)
        got = oracle.pack_k_row(u, d, bits)
        assert np.array_equal(got, want), (case["name"], np.flatnonzero(got != want)[:8])


def test_value_pair_rows_match_hand_derived_bytes(golden_dir):
    """One-hot value tokens packed into a pair row against hand-derived bytes: the
    channel permutation pos(c), the bit position inside the row, and which 16-bit half
    of each word the even and the odd token take."""
    d = 128
    for case in _golden_layout(golden_dir)["v_pairs"]:
        bits = case["bits"]
        u = np.zeros(d, np.uint8)
        u[case["channel"]] = case["code"]
        pairs = np.zeros(2 * d * bits // 8, np.uint8)
        oracle.pack_v_token(u, d, bits, 0 + case["odd"], pairs)
        want = np.zeros_like(pairs)
        for k, v in case["nonzero"].items():
            want[int(k)] = int(v, 16)
        assert np.array_equal(pairs, want), (case, np.flatnonzero(pairs)[:4], pairs[np.flatnonzero(pairs)[:4]])


def test_value_meta_records_match_hand_derived_bytes(golden_dir):
    """Value (scale, zero point) pairs of three tokens in the pair records, against records
    derived by hand: scales before zero points, the even token before the odd one, the
    odd half of the last record left 0."""
    case = _golden_layout(golden_dir)["v_meta"]
    d, bits, Gv = 128, case["bits"], case["Gv"]
    T = len(case["groups"])
    v = np.zeros((T, d), np.float64)
    for t, groups in enumerate(case["groups"]):
        for j, (lo, hi) in enumerate(groups):
            v[t, j * Gv:(j + 1) * Gv] = lo
            v[t, j * Gv + 1] = hi
    k = np.zeros((T, d), np.float16)
    st = oracle.cache_state(k, v.astype(np.float16), d=d, bits=bits, G=32, Gv=Gv, R=0)
    want = np.array([int(h, 16) for h in case["records"]], np.uint16)
    assert np.array_equal(st.v_meta.reshape(-1), want), [hex(x) for x in st.v_meta.reshape(-1)]


# ----------------------------------------------------------------------------- layout self-consistency
@pytest.mark.parametrize("bits", [2, 4, 8])
def test_layout_pack_unpack_round_trip(bits):
    d = 128
    rng = np.random.default_rng(bits)
    assert sorted(oracle.v_pos(d, c) for c in range(d)) == list(range(d))
    for _ in range(20):
        u = rng.integers(0, 2**bits, d).astype(np.uint8)
        assert np.array_equal(oracle.unpack_k_row(oracle.pack_k_row(u, d, bits), d, bits), u)
        pairs = np.zeros(4 * d * bits // 8, np.uint8)
        u2 = rng.integers(0, 2**bits, d).astype(np.uint8)
        oracle.pack_v_token(u, d, bits, 2, pairs)
        oracle.pack_v_token(u2, d, bits, 3, pairs)
        assert np.array_equal(oracle.unpack_v_token(pairs, d, bits, 2), u)
        assert np.array_equal(oracle.unpack_v_token(pairs, d, bits, 3), u2)
        assert not pairs[: 2 * d * bits // 8].any()


def test_cache_state_codes_agree_with_group_quantizer():
    rng = np.random.default_rng(12)
    d, T, G, Gv, bits = 128, 96, 32, 32, 2
    k16 = _f16(rng.standard_normal((T, d)))
    v16 = _f16(rng.standard_normal((T, d)))
    st = oracle.cache_state(k16, v16, d=d, bits=bits, G=G, Gv=Gv, R=0)
    for t in range(T):
        assert np.array_equal(oracle.unpack_v_token(st.v_codes, d, bits, t), st.v_u[t])
    for t in range(st.Tq):
        assert np.array_equal(oracle.unpack_k_row(st.k_codes[t], d, bits), st.k_u[t])
    # one key group by hand through the scalar quantizer
    g, c = 1, 77
    col = k16[g * G:(g + 1) * G, c]
    sh, zh = oracle.quant_params(col, bits)
    assert (st.k_meta[g, c, 0], st.k_meta[g, c, 1]) == (sh, zh)
    assert np.array_equal(st.k_u[g * G:(g + 1) * G, c], oracle.quantize_values(col, bits, sh, zh))


def test_mixed_width_state_is_the_two_single_width_states():
    """A cache with 8-bit keys and 4-bit values holds exactly the keys of the all-8-bit
    cache and the values of the all-4-bit cache (the two quantizers are independent)."""
    rng = np.random.default_rng(11)
    T, d = 300, 128
    k = (rng.standard_normal((T, d)) * 2).astype(np.float16)
    v = (rng.standard_normal((T, d)) * 0.5).astype(np.float16)
    mixed = oracle.cache_state(k, v, d=d, bits=8, G=32, Gv=64, R=128, v_bits=4)
    k8 = oracle.cache_state(k, v, d=d, bits=8, G=32, Gv=64, R=128)
    v4 = oracle.cache_state(k, v, d=d, bits=4, G=32, Gv=64, R=128)
    for name in ("k_codes", "k_meta", "k_resid", "k_u"):
        assert np.array_equal(getattr(mixed, name), getattr(k8, name)), name
    for name in ("v_codes", "v_meta", "v_u"):
        assert np.array_equal(getattr(mixed, name), getattr(v4, name)), name
    kh, vh = oracle.dequantize_state(mixed, d=d, bits=8, G=32, Gv=64, R=128, v_bits=4)
    kh8, _ = oracle.dequantize_state(k8, d=d, bits=8, G=32, Gv=64, R=128)
    _, vh4 = oracle.dequantize_state(v4, d=d, bits=4, G=32, Gv=64, R=128)
    assert np.array_equal(kh, kh8) and np.array_equal(vh, vh4)


# ----------------------------------------------------------------------------- symmetric scheme
# "KV Cache Quantization — 8-bit and 4-bit", § Symmetric vs asymmetric: zero point 0, the
# integer range centred on real zero, x_hat = scale * q; the -0.1 ... +3.0 example.

def test_symmetric_worked_example_wastes_the_negative_codes():
    """Data in [-0.1, 3.0]: the symmetric range must stretch to +-3.0. By hand:
    3.0/127 = 1.51181... * 2^-6; rounded up to 10 fraction bits: (1 + 525/1024) * 2^-6
    = 0.0236358642578125 (binary16 0x260D). -0.1 / scale = -4.23 -> q = -4; 3.0 / scale
    = 126.93 -> q = 127. So only the codes -4..127 (132 of 256) are ever used, while the
    asymmetric quantizer fitted to [-0.1, 3.0] spends all 256."""
    grid = np.unique(np.linspace(-0.1, 3.0, 20001).astype(np.float16))
    s = oracle.sym_params(grid, 8)
    assert s == 0x260D
    assert oracle.f32_from_f16(s) == 0.0236358642578125
    q = oracle.sym_quantize(grid, 8, s).astype(int) - 128
    assert q.min() == -4 and q.max() == 127
    assert len(np.unique(q)) == 132
    sa, za = oracle.quant_params(grid, 8)
    ua = oracle.quantize_values(grid, 8, sa, za)
    assert len(np.unique(ua)) == 256
    # the symmetric step is about twice the asymmetric one: twice the worst-case error
    assert 1.9 < oracle.f32_from_f16(s) / oracle.f32_from_f16(sa) < 2.0


def test_symmetric_round_trip_on_grid():
    """x = q * 2^-4 for every q in [-127, 127]: max|x| / 127 = 2^-4 exactly, so the
    stored scale is 2^-4 and every value comes back exactly."""
    q = np.arange(-127, 128)
    x = (q * 0.0625).astype(np.float16)
    s = oracle.sym_params(x, 8)
    assert s == 0x2C00  # 2^-4
    u = oracle.sym_quantize(x, 8, s)
    assert np.array_equal(u.astype(int) - 128, q)
    back = np.array([oracle.sym_dequantize_value(int(v), 8, s) for v in u])
    assert np.array_equal(back, x.astype(np.float64))


def test_symmetric_error_bound_and_odd_symmetry():
    """|x - x_hat| <= scale / 2 (the quotient x / scale is one binary32 rounding away
    from exact), no clipping (scale rounded up), and q(-x) = -q(x)."""
    rng = np.random.default_rng(5)
    for trial in range(200):
        n = int(rng.integers(1, 300))
        x = (rng.standard_normal(n) * 10.0 ** rng.uniform(-3, 3)).astype(np.float16)
        if trial % 7 == 0:
            x[rng.integers(n)] *= 40  # an outlier
        s = oracle.sym_params(x, 8)
        sf = oracle.f32_from_f16(s)
        u = oracle.sym_quantize(x, 8, s)
        q = u.astype(int) - 128
        assert q.min() >= -127 and q.max() <= 127
        xh = np.array([oracle.sym_dequantize_value(int(v), 8, s) for v in u])
        assert np.all(np.abs(x.astype(np.float64) - xh) <= sf / 2 * (1 + 2.0 ** -20))
        qn = oracle.sym_quantize(-x, 8, s).astype(int) - 128
        assert np.array_equal(qn, -q)


def test_symmetric_zero_vector():
    x = np.zeros(128, np.float16)
    s = oracle.sym_params(x, 8)
    assert s == 0x3C00
    u = oracle.sym_quantize(x, 8, s)
    assert np.all(u == 128)
    assert oracle.sym_dequantize_value(128, 8, s) == 0.0


def test_symmetric_cache_is_per_token():
    """Every token's keys and values carry their own scale: scaling one token's history
    leaves the other tokens' codes untouched, and every dequantized row is within half
    its own step of the input."""
    rng = np.random.default_rng(9)
    T, d = 37, 128
    k = (rng.standard_normal((T, d)) * 2).astype(np.float16)
    v = (rng.standard_normal((T, d)) * 0.5).astype(np.float16)
    st = oracle.cache_state_sym(k, v, d=d)
    assert st.Tq == T and st.k_meta.shape == (T,) and st.v_meta.shape == ((T + 1) // 2, 1, 4)
    assert np.all(oracle.value_meta(st)[:, 0, 1] == 0)
    assert np.all(st.v_meta[:, 0, 2:] == 0) and st.v_meta[-1, 0, 1] == 0  # zero points; token 37 does not exist
    k2 = k.copy()
    k2[5] *= np.float16(8)
    st2 = oracle.cache_state_sym(k2, v, d=d)
    others = np.arange(T) != 5
    assert np.array_equal(st2.k_u[others], st.k_u[others])
    assert np.array_equal(st2.k_u[5], st.k_u[5])  # a power-of-two rescale keeps the codes
    assert st2.k_meta[5] != st.k_meta[5]
    kh, vh = oracle.dequantize_state_sym(st, d=d)
    ks = np.array([oracle.f32_from_f16(int(h)) for h in st.k_meta])
    vs = np.array([oracle.f32_from_f16(int(h)) for h in oracle.value_meta(st)[:, 0, 0]])
    assert np.all(np.abs(k.astype(np.float64) - kh) <= ks[:, None] / 2 * (1 + 2.0 ** -20))
    assert np.all(np.abs(v.astype(np.float64) - vh) <= vs[:, None] / 2 * (1 + 2.0 ** -20))
    # the packed rows decode to the same codes
    for t in (0, 1, 36):
        assert np.array_equal(oracle.unpack_k_row(st.k_codes[t], d, 8), st.k_u[t])
        assert np.array_equal(oracle.unpack_v_token(st.v_codes.ravel(), d, 8, t), st.v_u[t])


# ----------------------------------------------------------------------------- outlier isolation
# "Sub-8-Bit KV Cache Quantization Is Not a Free Lever for an RDNA4 Agent Swarm", § What
# the low-bit numbers actually cost (per-vector dense-and-sparse quantization) and § The
# RDNA4 kernel angle (a sparse side channel). Reading: the k entries farthest from the
# vector's lower median, in order of distance, ties to the lower index.

def test_outlier_split_worked_example():
    """x = [1, 2, 3, 4, 50, 5, 6, -40]: sorted, the lower median (index 3) is 3; the
    distances are [2, 1, 0, 1, 47, 2, 3, 43], so the picks are 4 (50), 7 (-40), 6 (6),
    then the tie at distance 2 goes to channel 0 before channel 5."""
    x = np.array([1, 2, 3, 4, 50, 5, 6, -40], np.float16)
    idx, val, dense = oracle.split_outliers(x, 4)
    assert idx.tolist() == [4, 7, 6, 0]
    assert val.view(np.float16).tolist() == [50.0, -40.0, 6.0, 1.0]
    assert dense.view(np.float16).tolist() == [0, 2, 3, 4, 0, 5, 0, 0]
    idx0, _, dense0 = oracle.split_outliers(x, 0)
    assert idx0.size == 0 and np.array_equal(dense0, x.view(np.uint16))


def test_outlier_split_ties_and_two_values():
    """Ties in |x - median| go to the lower channel, and the median is the lower one:
    (a) 0.25 on 122 channels and +3 / -2.5 alternating on channels 10 .. 60: the median is
    0.25 and all six are 2.75 away, so the picks are channels 10, 20, 30, 40 in order;
    (b) 64 channels at -2 and 64 at +2: the lower median is -2, every +2 is 4 away, so
    the picks are the four lowest +2 channels; (c) a constant row: every distance is 0,
    so channels 0 .. 3, and the dense row keeps the constant elsewhere."""
    x = np.full(128, 0.25, np.float16)
    x[[10, 20, 30, 40, 50, 60]] = [3.0, -2.5, 3.0, -2.5, 3.0, -2.5]
    idx, val, dense = oracle.split_outliers(x, 4)
    assert idx.tolist() == [10, 20, 30, 40]
    assert val.view(np.float16).tolist() == [3.0, -2.5, 3.0, -2.5]
    assert dense.view(np.float16)[[10, 20, 30, 40, 50, 60]].tolist() == [0, 0, 0, 0, 3.0, -2.5]
    x = np.full(128, 2.0, np.float16)
    neg = np.random.default_rng(5).permutation(128)[:64]
    x[neg] = -2.0
    pos = sorted(set(range(128)) - set(neg.tolist()))
    idx, val, _ = oracle.split_outliers(x, 4)
    assert idx.tolist() == pos[:4]
    assert val.view(np.float16).tolist() == [2.0] * 4
    x = np.full(128, 1.5, np.float16)
    idx, val, dense = oracle.split_outliers(x, 3)
    assert idx.tolist() == [0, 1, 2]
    assert dense.view(np.float16).tolist() == [0.0] * 3 + [1.5] * 125


def test_outliers_shrink_the_dense_scale():
    """A key row with three planted outliers: they are the three picks, their values come
    back exactly, and the dense scale drops to max|rest| / 127 (rounded up), so every
    other channel is within half of that smaller step."""
    rng = np.random.default_rng(21)
    x = rng.standard_normal(128).astype(np.float16)
    planted = [5, 77, 120]
    x[planted] = np.array([40.0, -35.0, 52.0], np.float16)
    T = 1
    st0 = oracle.cache_state_sym(x[None, :], x[None, :], d=128)
    st = oracle.cache_state_sym(x[None, :], x[None, :], d=128, k_outliers=3)
    assert sorted(st.k_sparse[0, :, 0].tolist()) == planted
    rest = np.delete(x.astype(np.float32), planted)
    assert st.k_meta[0] == oracle.f16_from_f32_ru(float(np.abs(rest).max() / np.float32(127)))
    assert oracle.f32_from_f16(int(st.k_meta[0])) < oracle.f32_from_f16(int(st0.k_meta[0])) / 10
    kh, _ = oracle.dequantize_state_sym(st, d=128)
    assert np.array_equal(kh[0, planted], x[planted].astype(np.float32))
    s = oracle.f32_from_f16(int(st.k_meta[0]))
    others = np.setdiff1d(np.arange(128), planted)
    assert np.all(np.abs(kh[0, others] - x[others].astype(np.float64)) <= s / 2 * (1 + 2.0 ** -20))
    assert T == 1


def test_outliers_cut_the_error_on_outlier_channels():
    """Keys with planted outlier channels (the benchmark generator's a*z + 5 on 4
    channels): isolating 4 entries per row lowers the worst error of the other channels
    by more than 10x and leaves the isolated ones exact."""
    import synth
    w = synth.WORKLOADS["sym8-b16"]
    T = 64
    k = synth.k_slice(w, 0, 0, 0, range(T))
    v = synth.v_slice(w, 0, 0, 0, range(T))
    e0 = np.abs(oracle.dequantize_state_sym(oracle.cache_state_sym(k, v, d=128), d=128)[0] - k.astype(np.float64))
    st = oracle.cache_state_sym(k, v, d=128, k_outliers=4)
    e4 = np.abs(oracle.dequantize_state_sym(st, d=128)[0] - k.astype(np.float64))
    assert e4.max() * 10 < e0.max()
    for t in range(T):
        assert np.all(e4[t, st.k_sparse[t, :, 0]] == 0)


# ----------------------------------------------------------------------------- outliers with per-channel keys
def test_per_channel_keys_with_isolated_entries():
    """Per-channel keys with k isolated entries per key row ("Sub-8-Bit KV Cache Quantization
    Is Not a Free Lever for an RDNA4 Agent Swarm", § What the low-bit numbers actually cost:
    dense-and-sparse). Two planted channels far from every row's median are the isolated
    entries of every quantized row, in order of distance, with their exact binary16 values;
    their dense columns are all +0, so their groups get scale 1 and zero point q_min; every
    other channel's group parameters are those of its untouched column; dequantized keys
    are exact on the isolated channels and within half a stored step elsewhere; residual
    rows stay whole and the split of a row does not depend on later tokens."""
    rng = np.random.default_rng(4242)
    d, G, R, Gv = 128, 32, 64, 64
    T = 3 * R + 20
    big = (7, 91)
    for bits in (8, 4, 2):
        k = rng.standard_normal((T, d)).astype(np.float16)
        k[:, big[0]] = (1000 + 50 * rng.standard_normal(T)).astype(np.float16)
        k[:, big[1]] = (-2000 + 50 * rng.standard_normal(T)).astype(np.float16)
        v = rng.standard_normal((T, d)).astype(np.float16)
        st = oracle.cache_state(k, v, d=d, bits=bits, G=G, Gv=Gv, R=R, k_outliers=2)
        Tq = st.Tq
        assert Tq == 3 * R and st.k_sparse.shape == (Tq, 2, 2)
        assert (st.k_sparse[:, 0, 0] == big[1]).all() and (st.k_sparse[:, 1, 0] == big[0]).all()
        assert np.array_equal(st.k_sparse[:, 0, 1], k[:Tq, big[1]].view(np.uint16))
        assert np.array_equal(st.k_sparse[:, 1, 1], k[:Tq, big[0]].view(np.uint16))
        qmin_bits = int(np.float16(oracle.qmin(bits)).view(np.uint16))
        for g in range(Tq // G):
            for c in range(d):
                if c in big:
                    assert tuple(st.k_meta[g, c]) == (0x3C00, qmin_bits), (bits, g, c)
                else:
                    assert tuple(st.k_meta[g, c]) == oracle.quant_params(k[g * G:(g + 1) * G, c], bits), (bits, g, c)
        kh, _ = oracle.dequantize_state(st, d=d, bits=bits, G=G, Gv=Gv, R=R)
        for c in big:
            assert np.array_equal(kh[:Tq, c], k[:Tq, c].astype(np.float32))
        scales = st.k_meta[:, :, 0].view(np.float16).astype(np.float64)  # [group][channel]
        err = np.abs(kh[:Tq].astype(np.float64) - k[:Tq].astype(np.float64))
        bound = np.repeat(scales, G, axis=0) / 2 * (1 + 2.0**-20)
        assert (err <= bound).all()
        assert np.array_equal(st.k_resid[:T - Tq], k[Tq:].view(np.uint16))
        assert np.array_equal(kh[Tq:], k[Tq:].astype(np.float32))
        st2 = oracle.cache_state(k[:2 * R + 5], v[:2 * R + 5], d=d, bits=bits, G=G, Gv=Gv, R=R, k_outliers=2)
        assert np.array_equal(st2.k_sparse, st.k_sparse[:st2.Tq])
