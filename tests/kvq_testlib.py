"""Shared helpers of the parity tests: slices of the GPU cache buffers, oracle
states of the same slices, and element-by-element comparisons.

Inputs come from the seeded generator (host numpy side for the oracle, device
side or host copies for the CUDA side); expected values come from ``oracle`` only.
"""

from __future__ import annotations

import math

import numpy as np

import oracle
import synth

ATOL = 2e-3  # decode attention: max-abs error against the oracle's attention over x_hat


def cfg_dims(cache):
    c = cache.cfg
    sym = int(c.symmetric)
    R_eff = 1 if sym else (c.residual_len if c.residual_len > 0 else c.k_group)
    S_pad = (c.max_seq_len + 127) // 128 * 128
    row = c.d_head * c.bits // 8
    vbits = c.v_bits or c.bits
    return dict(L=c.n_layers, B=c.batch, H=c.n_kv_heads, r=c.gqa_ratio, d=c.d_head, bits=c.bits, vbits=vbits,
                rowV=c.d_head * vbits // 8, G=c.k_group,
                Gv=c.v_group, R=c.residual_len, R_eff=R_eff, S_pad=S_pad, row=row, n_vg=c.d_head // c.v_group,
                sym=sym, kout=int(c.k_outliers))


def gpu_slice_state(cache, layer: int, b: int, h: int, T: int):
    """The five buffers of one (layer, b, h) slice, cut to the valid part for T tokens (numpy)."""
    import torch  # noqa: F401

    g = cfg_dims(cache)
    sl = (layer * g["B"] + b) * g["H"] + h
    Tq = (T // g["R_eff"]) * g["R_eff"]

    def part(name, slice_bytes, nbytes):
        buf = cache.buffer(name)
        return buf[sl * slice_bytes: sl * slice_bytes + nbytes].cpu().numpy()

    kc = part("k_codes", g["S_pad"] * g["row"], Tq * g["row"]).reshape(Tq, g["row"])
    ksp = None
    if g["sym"]:  # one binary16 key scale per token (then the isolated entries), no residual window
        km_slice = g["S_pad"] * 2 + g["S_pad"] * g["kout"] * 4
        km = part("k_meta", km_slice, Tq * 2).view(np.uint16).reshape(Tq)
        if g["kout"]:
            buf = cache.buffer("k_meta")
            off = sl * km_slice + g["S_pad"] * 2
            ksp = buf[off: off + Tq * g["kout"] * 4].cpu().numpy().view(np.uint16).reshape(Tq, g["kout"], 2)
        kr = np.zeros((0, g["d"]), np.uint16)
    else:
        km_groups = (g["S_pad"] // g["G"]) * g["d"] * 4
        km_slice = km_groups + g["S_pad"] * g["kout"] * 4
        km = part("k_meta", km_slice, (Tq // g["G"]) * g["d"] * 4).view(np.uint16)
        km = km.reshape(Tq // g["G"], g["d"], 2)
        if g["kout"]:  # isolated entries of the quantized rows, after the groups' metadata
            buf = cache.buffer("k_meta")
            off = sl * km_slice + km_groups
            ksp = buf[off: off + Tq * g["kout"] * 4].cpu().numpy().view(np.uint16).reshape(Tq, g["kout"], 2)
        kr = part("k_resid", g["R_eff"] * g["d"] * 2, (T - Tq) * g["d"] * 2).view(np.uint16).reshape(T - Tq, g["d"])
    npairs = (T + 1) // 2
    vc = part("v_codes", g["S_pad"] * g["rowV"], npairs * 2 * g["rowV"]).reshape(npairs, 2 * g["rowV"])
    vm = part("v_meta", g["S_pad"] * g["n_vg"] * 4, npairs * g["n_vg"] * 8).view(np.uint16).reshape(npairs, g["n_vg"], 4)
    return dict(k_codes=kc, k_meta=km, k_resid=kr, v_codes=vc, v_meta=vm, Tq=Tq, k_sparse=ksp)


def oracle_slice_state(k_hist, v_hist, cache):
    g = cfg_dims(cache)
    if g["sym"]:
        return oracle.cache_state_sym(k_hist, v_hist, d=g["d"], k_outliers=g["kout"])
    return oracle.cache_state(k_hist, v_hist, d=g["d"], bits=g["bits"], G=g["G"], Gv=g["Gv"], R=g["R"],
                              v_bits=g["vbits"], k_outliers=g["kout"])


def assert_slice_equal(gpu: dict, st: oracle.OracleState, where: str = ""):
    T = st.T
    assert gpu["Tq"] == st.Tq
    if st.k_sparse is not None and st.k_sparse.size:
        if not np.array_equal(gpu["k_sparse"], st.k_sparse):
            bad = np.argwhere(gpu["k_sparse"] != st.k_sparse)
            raise AssertionError(f"{where} k_sparse: {len(bad)} mismatches, first at {bad[:3].tolist()}")
    for name in ("k_codes", "k_meta", "v_codes", "v_meta"):
        a, e = gpu[name], getattr(st, name)
        assert a.shape == e.shape, (where, name, a.shape, e.shape)
        if not np.array_equal(a, e):
            bad = np.argwhere(a != e)
            raise AssertionError(f"{where} {name}: {len(bad)} mismatches, first at {bad[:3].tolist()}")
    n_res = T - st.Tq
    if n_res == 0 and gpu["k_resid"].size == 0:
        return
    R_eff = st.k_resid.shape[0]
    # residual slot (t mod R_eff) of tokens [Tq, T); with Tq a multiple of R_eff that is t - Tq
    exp_res = st.k_resid[:n_res] if n_res <= R_eff else None
    assert exp_res is not None
    if not np.array_equal(gpu["k_resid"], exp_res):
        raise AssertionError(f"{where} k_resid mismatch")


def oracle_attention(st: oracle.OracleState, q_rows, cache, softmax_scale):
    g = cfg_dims(cache)
    if g["sym"]:
        kh, vh = oracle.dequantize_state_sym(st, d=g["d"])
    else:
        kh, vh = oracle.dequantize_state(st, d=g["d"], bits=g["bits"], G=g["G"], Gv=g["Gv"], R=g["R"],
                                         v_bits=g["vbits"])
    return oracle.attention(q_rows, kh, vh, softmax_scale)


def small_workload(name="small", *, L=1, H=2, r=4, B=2, S=600, steps=8, bits=4, G=32, Gv=64, R=128, n_out=2,
                   gain=20, seed=777, v_bits=0, symmetric=0, k_outliers=0):
    return synth.Workload(name, L, H, r, 128, B, S, steps, bits, G, Gv, R, n_out, gain, seed, v_bits=v_bits,
                          symmetric=symmetric, k_outliers=k_outliers)


def host_layer_inputs(w, layer, t0, nt):
    """Keys and values [B][nt][H][d] of tokens [t0, t0+nt) from the host generator."""
    toks = np.arange(t0, t0 + nt)
    k = synth.gen_k(w.seed, layer, range(w.batch), toks, w.n_kv, w.d_head, w.n_out, w.gain, w.shift)
    v = synth.gen_v(w.seed, layer, range(w.batch), toks, w.n_kv, w.d_head)
    return k, v


def softmax_scale(w):
    return 1.0 / math.sqrt(w.d_head)


def oracle_slice_job(job):
    """Oracle side of one (layer, batch row, kv head) slice of a full-size workload, for a
    process pool: the packed state after each T in `job["Ts"]` (the state after the last T
    is returned in full) and the oracle attention of the query rows given for each T.
    Runs in a worker process (spawned, no CUDA); inputs come from the host generator."""
    w, layer, b, h = job["w"], job["layer"], job["b"], job["h"]
    T_max = max(job["Ts"])
    k = synth.k_slice(w, layer, b, h, range(T_max))
    v = synth.v_slice(w, layer, b, h, range(T_max))
    out = {"key": (layer, b, h), "att": {}}
    for T in job["Ts"]:
        if w.symmetric:
            st = oracle.cache_state_sym(k[:T], v[:T], d=w.d_head, k_outliers=w.k_outliers)
            kh, vh = oracle.dequantize_state_sym(st, d=w.d_head)
        else:
            st = oracle.cache_state(k[:T], v[:T], d=w.d_head, bits=w.bits, G=w.k_group, Gv=w.v_group, R=w.residual,
                                    v_bits=w.vbits, k_outliers=w.k_outliers)
            kh, vh = oracle.dequantize_state(st, d=w.d_head, bits=w.bits, G=w.k_group, Gv=w.v_group, R=w.residual,
                                             v_bits=w.vbits)
        if T in job["q"]:
            out["att"][T] = oracle.attention(job["q"][T], kh, vh, w.softmax_scale)
        if T == T_max:
            out["state"] = st
    return out
