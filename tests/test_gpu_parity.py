"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Codes, scales, zero points and the residual window must match bit for bit;
dequantized values bit for bit; decode attention within 2e-3 max-abs.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from kvq_testlib import (ATOL, assert_slice_equal, gpu_slice_state, host_layer_inputs,  # noqa: E402
                         oracle_attention, oracle_slice_state, small_workload, softmax_scale)

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from bit_kv_cache_09_gb300 import kvq  # noqa: E402
from bit_kv_cache_09_gb300.cache import QuantizedKVCache  # noqa: E402

IMPLS = [kvq.DECODE_SIMT, kvq.DECODE_MMA]


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _history(w, layer, b, h, T):
    return synth.k_slice(w, layer, b, h, range(T)), synth.v_slice(w, layer, b, h, range(T))


def _check_all_slices(cache, w, layer, T, k_host, v_host):
    """Bit-exact state of every (b, h) slice after T tokens; k_host/v_host [B][T][H][d]."""
    for b in range(w.batch):
        for h in range(w.n_kv):
            st = oracle_slice_state(k_host[b, :T, h], v_host[b, :T, h], cache)
            assert_slice_equal(gpu_slice_state(cache, layer, b, h, T), st, f"b={b} h={h} T={T}")


def _check_attention(cache, w, layer, T, k_host, v_host, q_host, impl):
    q = _dev(q_host)
    out = cache.attention(layer, T, q, softmax_scale(w), impl=impl).cpu().numpy()
    worst = 0.0
    for b in range(w.batch):
        for h in range(w.n_kv):
            st = oracle_slice_state(k_host[b, :T, h], v_host[b, :T, h], cache)
            ref = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
            got = out[b, h * w.gqa:(h + 1) * w.gqa]
            worst = max(worst, float(np.abs(got - ref).max()))
    assert worst <= ATOL, worst
    return worst


def test_device_generator_matches_host():
    from synth.device import DeviceGenerator

    for name in ("tiny-int8", "kivi-int2", "long-int4-16k"):
        w = synth.WORKLOADS[name]
        gen = DeviceGenerator(w)
        k, v = gen.kv(layer=3 % w.n_layers, t0=1000, nt=40, b0=0, nb=2)
        kh = synth.gen_k(w.seed, 3 % w.n_layers, [0, 1], range(1000, 1040), w.n_kv, w.d_head, w.n_out, w.gain)
        vh = synth.gen_v(w.seed, 3 % w.n_layers, [0, 1], range(1000, 1040), w.n_kv, w.d_head)
        assert np.array_equal(k.cpu().numpy().view(np.uint16), kh.view(np.uint16))
        assert np.array_equal(v.cpu().numpy().view(np.uint16), vh.view(np.uint16))
        q = gen.q(layer=0, step_token=w.seq + 5, b0=1, nb=1)
        qh = synth.gen_q(w.seed, 0, [1], w.seq + 5, w.n_q, w.d_head)
        assert np.array_equal(q.cpu().numpy().view(np.uint16), qh.view(np.uint16))


@pytest.mark.parametrize("impl", IMPLS)
def test_tiny_workload_full_parity(impl):
    """One layer, one kv head, GQA 4, int8, K groups of 32, no residual; prefill of 256
    tokens and one decode step: every byte of the cache, every dequantized value and
    every attention output."""
    w = synth.WORKLOADS["tiny-int8"]
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.seq + w.steps)
    cache.append(0, 0, _dev(k_host[:, :w.seq]), _dev(v_host[:, :w.seq]))
    _check_all_slices(cache, w, 0, w.seq, k_host, v_host)
    q0 = synth.gen_q(w.seed, 0, range(w.batch), w.seq - 1, w.n_q, w.d_head)
    _check_attention(cache, w, 0, w.seq, k_host, v_host, q0, impl)
    for s in range(w.steps):
        T = w.seq + s
        cache.append(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]))
        _check_all_slices(cache, w, 0, T + 1, k_host, v_host)
        q = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        _check_attention(cache, w, 0, T + 1, k_host, v_host, q, impl)
    # dequantize: bit-exact against the oracle's binary32 x_hat
    T = w.seq + w.steps
    kd, vd = cache.dequantize(0, T)
    st = oracle_slice_state(k_host[0, :T, 0], v_host[0, :T, 0], cache)
    kh, vh = oracle.dequantize_state(st, d=128, bits=w.bits, G=w.k_group, Gv=w.v_group, R=w.residual)
    assert np.array_equal(kd[0, 0].cpu().numpy().view(np.uint32), kh.view(np.uint32))
    assert np.array_equal(vd[0, 0].cpu().numpy().view(np.uint32), vh.view(np.uint32))


CONFIGS = [
    # bits, G, Gv, R, r
    (8, 32, 128, 0, 4),
    (8, 128, 128, 0, 4),
    (4, 128, 64, 128, 4),
    (2, 32, 32, 128, 4),
    (4, 128, 128, 128, 8),
    (4, 64, 32, 256, 3),
    (2, 128, 64, 0, 1),
    (2, 64, 128, 128, 4),   # 2-bit values in groups of 128 channels (four lanes per group)
    (4, 32, 64, 64, 2),     # 4-bit keys in groups of 32 tokens (one warp per group)
]


@pytest.mark.parametrize("bits,G,Gv,R,r", CONFIGS)
@pytest.mark.parametrize("impl", IMPLS)
def test_ragged_prefill_decode_and_flush(bits, G, Gv, R, r, impl):
    """Prefill of a ragged length, then decode steps that cross a residual flush."""
    R_eff = R if R > 0 else G
    off = min(37, R_eff - 5)
    S = 3 * R_eff + off  # ragged: several tiles plus a partial residual
    steps = R_eff - off + 3  # crosses the next flush
    w = small_workload(bits=bits, G=G, Gv=Gv, R=R, r=r, B=2, H=2, S=S, steps=steps, seed=1000 + bits * 10 + r)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    cache.append(0, 0, _dev(k_host[:, :S]), _dev(v_host[:, :S]))
    _check_all_slices(cache, w, 0, S, k_host, v_host)
    for s in range(steps):
        T = S + s
        cache.append(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]))
        if s in (0, steps - 4, steps - 3, steps - 1):
            _check_all_slices(cache, w, 0, T + 1, k_host, v_host)
            q = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
            _check_attention(cache, w, 0, T + 1, k_host, v_host, q, impl)


def test_chunked_appends_equal_one_shot():
    """The cache state depends only on the token history, not on how it was appended."""
    w = small_workload(bits=4, G=32, Gv=64, R=128, B=2, H=3, S=650, steps=0, seed=4242)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.seq)
    rng = np.random.default_rng(0)
    cache = QuantizedKVCache.for_workload(w)
    T = 0
    while T < w.seq:
        n = int(min(w.seq - T, rng.integers(1, 150)))
        cache.append(0, T, _dev(k_host[:, T:T + n]), _dev(v_host[:, T:T + n]))
        T += n
        if rng.random() < 0.3:
            _check_all_slices(cache, w, 0, T, k_host, v_host)
    _check_all_slices(cache, w, 0, T, k_host, v_host)


def test_layers_are_independent():
    w = small_workload(L=3, bits=2, G=32, Gv=32, R=128, B=1, H=2, S=300, steps=0, seed=99)
    cache = QuantizedKVCache.for_workload(w)
    ins = {}
    for layer in (2, 0):
        k_host, v_host = host_layer_inputs(w, layer, 0, w.seq)
        ins[layer] = (k_host, v_host)
        cache.append(layer, 0, _dev(k_host), _dev(v_host))
    for layer in (0, 2):
        _check_all_slices(cache, w, layer, w.seq, *ins[layer])
    g = cache.buffer("k_codes")
    n = g.numel() // 3
    assert not g[n:2 * n].any()  # layer 1 untouched


@pytest.mark.parametrize("bits,G,Gv,R,r", [(8, 128, 128, 0, 4), (4, 128, 64, 128, 4), (2, 32, 32, 128, 4),
                                          (4, 128, 128, 128, 8), (4, 64, 32, 256, 3)])
def test_fused_decode_step(bits, G, Gv, R, r):
    """kvq_decode_step (append fused into the attention launch) leaves the same cache
    state as the oracle and gives the same outputs as the two separate calls, across a
    residual flush (where it takes the two-launch path)."""
    R_eff = R if R > 0 else G
    S = 2 * R_eff + 7
    steps = R_eff - 7 + 4
    w = small_workload(bits=bits, G=G, Gv=Gv, R=R, r=r, B=3, H=2, S=S, steps=steps, seed=2000 + bits + r)
    fused = QuantizedKVCache.for_workload(w)
    split = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    for c in (fused, split):
        c.append(0, 0, _dev(k_host[:, :S]), _dev(v_host[:, :S]))
    for s in range(steps):
        T = S + s
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        kd, vd, qd = _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host)
        out_f = fused.decode_step(0, T, kd, vd, qd, softmax_scale(w))
        split.append(0, T, kd, vd)
        out_s = split.attention(0, T + 1, qd, softmax_scale(w))
        assert torch.equal(out_f, out_s), (s, (out_f - out_s).abs().max().item())
        if s in (0, 1, steps - 5, steps - 4, steps - 1):
            _check_all_slices(fused, w, 0, T + 1, k_host, v_host)
            _check_attention(fused, w, 0, T + 1, k_host, v_host, q_host, kvq.DECODE_AUTO)


def _all_f16_values():
    """Every finite binary16 value, as float64, sorted, with its bit pattern."""
    bits = np.arange(0x10000, dtype=np.uint32).astype(np.uint16)
    with np.errstate(invalid="ignore"):
        vals = bits.view(np.float16).astype(np.float64)
    ok = np.isfinite(vals)
    order = np.argsort(vals[ok], kind="stable")
    return vals[ok][order], bits[ok][order]


def _near_midpoints(lo, hi, s, n, vals, bits):
    """n binary16 values strictly inside (lo, hi) whose quotient by s is closest to a
    half-integer (where a wrongly rounded division would change the code)."""
    a, b = np.searchsorted(vals, lo, side="right"), np.searchsorted(vals, hi, side="left")
    cand_v, cand_b = vals[a:b], bits[a:b]
    if cand_v.size == 0:
        return np.zeros(0, np.uint16)
    t = cand_v / s
    dist = np.abs(t - np.floor(t) - 0.5)
    return cand_b[np.argsort(dist, kind="stable")[:n]]


@pytest.mark.parametrize("bits", [8, 4, 2])
def test_quantize_near_rounding_midpoints(bits):
    """Inputs planted where x / scale is as close as binary16 allows to a half-integer:
    the kernels' fma-corrected division must give the same codes as the oracle's IEEE
    division (prefill through the key-group and value-token kernels, then decode steps
    through the fused append)."""
    G = Gv = 32
    w = small_workload(bits=bits, G=G, Gv=Gv, R=0, r=4, B=1, H=1, S=64, steps=6, seed=4100 + bits)
    vals, pats = _all_f16_values()
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    k_host, v_host = k_host.copy(), v_host.copy()
    kb, vb = k_host.view(np.uint16), v_host.view(np.uint16)
    rng = np.random.default_rng(bits)
    # keys: per group of G tokens and channel, overwrite 8 tokens that are neither the min nor the max
    for g0 in range(0, 64, G):
        for c in range(128):
            col = k_host[0, g0:g0 + G, 0, c].astype(np.float64)
            s_h, _ = oracle.quant_params(k_host[0, g0:g0 + G, 0, c], bits)
            s = float(np.array([s_h], np.uint16).view(np.float16)[0])
            pick = _near_midpoints(col.min(), col.max(), s, 8, vals, pats)
            inner = [t for t in rng.permutation(G) if col[t] != col.min() and col[t] != col.max()][:pick.size]
            for t, pb in zip(inner, pick):
                kb[0, g0 + t, 0, c] = pb
    # values: per token and group of Gv channels, overwrite 6 inner channels
    for t in range(w.max_seq):
        for g0 in range(0, 128, Gv):
            row = v_host[0, t, 0, g0:g0 + Gv].astype(np.float64)
            s_h, _ = oracle.quant_params(v_host[0, t, 0, g0:g0 + Gv], bits)
            s = float(np.array([s_h], np.uint16).view(np.float16)[0])
            pick = _near_midpoints(row.min(), row.max(), s, 6, vals, pats)
            inner = [c for c in rng.permutation(Gv) if row[c] != row.min() and row[c] != row.max()][:pick.size]
            for c, pb in zip(inner, pick):
                vb[0, t, 0, g0 + c] = pb
    cache = QuantizedKVCache.for_workload(w)
    cache.append(0, 0, _dev(k_host[:, :64]), _dev(v_host[:, :64]))
    _check_all_slices(cache, w, 0, 64, k_host, v_host)
    for s in range(w.steps):
        T = 64 + s
        q = _dev(synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head))
        cache.decode_step(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), q, softmax_scale(w))
    _check_all_slices(cache, w, 0, 64 + w.steps, k_host, v_host)


@pytest.mark.parametrize("bits,G,Gv,R,r", [(8, 128, 128, 0, 4), (4, 128, 64, 128, 8), (2, 32, 32, 128, 3)])
def test_small_grid_long_sequence(bits, G, Gv, R, r):
    """Two (batch row, kv head) pairs over ~4k tokens: the plan runs each pair as one
    16-CTA cluster of 8-warp CTAs (each warp then owns one 32-token iteration), through
    both the attention call and the fused decode step."""
    w = small_workload(bits=bits, G=G, Gv=Gv, R=R, r=r, B=1, H=2, S=3900, steps=3, seed=5000 + bits + r)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    cache.append(0, 0, _dev(k_host[:, :w.seq]), _dev(v_host[:, :w.seq]))
    q0 = synth.gen_q(w.seed, 0, range(w.batch), w.seq - 1, w.n_q, w.d_head)
    _check_attention(cache, w, 0, w.seq, k_host, v_host, q0, kvq.DECODE_MMA)
    for s in range(w.steps):
        T = w.seq + s
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        out = cache.decode_step(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host),
                                softmax_scale(w)).cpu().numpy()
        for h in range(w.n_kv):
            st = oracle_slice_state(k_host[0, :T + 1, h], v_host[0, :T + 1, h], cache)
            ref = oracle_attention(st, q_host[0, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
            assert float(np.abs(out[0, h * w.gqa:(h + 1) * w.gqa] - ref).max()) <= ATOL
    _check_all_slices(cache, w, 0, w.max_seq, k_host, v_host)


MIXED = [
    # G, Gv, R, r  (8-bit keys, 4-bit values)
    (128, 64, 128, 4),
    (32, 128, 0, 4),
    (64, 32, 256, 3),
    (128, 128, 128, 8),
    (32, 64, 128, 1),
]


@pytest.mark.parametrize("G,Gv,R,r", MIXED)
def test_mixed_widths_prefill_decode_flush_and_dequantize(G, Gv, R, r):
    """8-bit keys with 4-bit values: a ragged prefill, decode steps across a residual
    flush (attention call and fused step on two caches), and the dequantized history,
    all against the oracle run with the same two widths."""
    R_eff = R if R > 0 else G
    off = min(37, R_eff - 5)
    S = 3 * R_eff + off
    steps = R_eff - off + 3
    w = small_workload(bits=8, v_bits=4, G=G, Gv=Gv, R=R, r=r, B=2, H=2, S=S, steps=steps, seed=6100 + G + r)
    split = QuantizedKVCache.for_workload(w)
    fused = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    for c in (split, fused):
        c.append(0, 0, _dev(k_host[:, :S]), _dev(v_host[:, :S]))
    _check_all_slices(split, w, 0, S, k_host, v_host)
    for s in range(steps):
        T = S + s
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        kd, vd, qd = _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host)
        out_f = fused.decode_step(0, T, kd, vd, qd, softmax_scale(w))
        split.append(0, T, kd, vd)
        out_s = split.attention(0, T + 1, qd, softmax_scale(w), impl=kvq.DECODE_MMA)
        assert torch.equal(out_f, out_s), (s, (out_f - out_s).abs().max().item())
        if s in (0, steps - 4, steps - 3, steps - 1):
            _check_all_slices(fused, w, 0, T + 1, k_host, v_host)
            _check_attention(split, w, 0, T + 1, k_host, v_host, q_host, kvq.DECODE_MMA)
    T = S + steps
    kd, vd = split.dequantize(0, T)
    for b in range(w.batch):
        for h in range(w.n_kv):
            st = oracle_slice_state(k_host[b, :T, h], v_host[b, :T, h], split)
            kh, vh = oracle.dequantize_state(st, d=128, bits=8, G=G, Gv=Gv, R=R, v_bits=4)
            assert np.array_equal(kd[b, h].cpu().numpy().view(np.uint32), kh.view(np.uint32))
            assert np.array_equal(vd[b, h].cpu().numpy().view(np.uint32), vh.view(np.uint32))


def test_mixed_widths_small_grid_long_sequence():
    """8-bit keys with 4-bit values over ~4k tokens for two pairs (16-CTA clusters of
    8-warp CTAs)."""
    w = small_workload(bits=8, v_bits=4, G=128, Gv=64, R=128, r=4, B=1, H=2, S=3900, steps=2, seed=6500)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    cache.append(0, 0, _dev(k_host[:, :w.seq]), _dev(v_host[:, :w.seq]))
    q0 = synth.gen_q(w.seed, 0, range(w.batch), w.seq - 1, w.n_q, w.d_head)
    _check_attention(cache, w, 0, w.seq, k_host, v_host, q0, kvq.DECODE_MMA)
    _check_attention(cache, w, 0, w.seq, k_host, v_host, q0, kvq.DECODE_AUTO)


def test_mixed_widths_have_no_simt_path():
    """The scalar decode path handles one code width only; a mixed cache asks for the
    tensor-core path and gets an UNSUPPORTED status from the scalar one."""
    w = small_workload(bits=8, v_bits=4, G=32, Gv=64, R=128, B=1, H=1, S=40, steps=0, seed=1)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.seq)
    cache.append(0, 0, _dev(k_host), _dev(v_host))
    q = _dev(synth.gen_q(w.seed, 0, range(1), w.seq - 1, w.n_q, w.d_head))
    with pytest.raises(kvq.KVQError):
        cache.attention(0, w.seq, q, softmax_scale(w), impl=kvq.DECODE_SIMT)


@pytest.mark.parametrize("bits,v_bits,G,Gv,R,B,H,S", [
    (4, 0, 128, 64, 128, 32, 4, 2049),
    (4, 0, 64, 64, 128, 32, 4, 2049),  # 64-token key groups on the 8-warp key kernel (full grid)
    (2, 0, 32, 32, 128, 32, 4, 2049),
    (8, 4, 128, 64, 128, 12, 4, 4000),
    (8, 0, 128, 128, 0, 12, 4, 4000),
])
def test_large_grid(bits, v_bits, G, Gv, R, B, H, S):
    """Grids of 48 or 128 (batch row, kv head) pairs (the large-grid split plans: several
    splits per pair, merged in clusters or through the workspace): attention call and
    fused decode step against the oracle for every pair."""
    w = small_workload(bits=bits, v_bits=v_bits, G=G, Gv=Gv, R=R, r=4, B=B, H=H, S=S, steps=3,
                       seed=7000 + bits + v_bits + B)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    cache.append(0, 0, _dev(k_host[:, :S]), _dev(v_host[:, :S]))
    assert kvq.kvq_decode_num_splits(cache.cfg, S) > 1
    q0 = synth.gen_q(w.seed, 0, range(w.batch), S - 1, w.n_q, w.d_head)
    _check_attention(cache, w, 0, S, k_host, v_host, q0, kvq.DECODE_MMA)
    for s in range(w.steps):
        T = S + s
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        out = cache.decode_step(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host),
                                softmax_scale(w)).cpu().numpy()
        if s == w.steps - 1:
            worst = 0.0
            for b in range(w.batch):
                for h in range(w.n_kv):
                    st = oracle_slice_state(k_host[b, :T + 1, h], v_host[b, :T + 1, h], cache)
                    ref = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
                    worst = max(worst, float(np.abs(out[b, h * w.gqa:(h + 1) * w.gqa] - ref).max()))
            assert worst <= ATOL, worst
    _check_all_slices(cache, w, 0, S + w.steps, k_host, v_host)


SYM_CASES = [
    # r, B, H, S, steps
    (4, 2, 2, 300, 5),     # small grid, 4-warp clusters
    (8, 2, 2, 257, 4),     # GQA 8
    (4, 1, 2, 3900, 2),    # small grid over ~4k tokens (8-warp clusters)
    (4, 12, 4, 2100, 2),   # large grid (split plan)
]


@pytest.mark.parametrize("r,B,H,S,steps", SYM_CASES)
def test_symmetric_per_token_int8(r, B, H, S, steps):
    """Symmetric per-token int8 keys and values: a prefill in two chunks, decode steps
    through kvq_decode_step, every slice bit-exact (codes, per-token scales, value
    meta), attention within 2e-3 and the dequantized history bit-exact against the
    oracle; the CUDA-core kernel declines the scheme."""
    w = small_workload(bits=8, G=128, Gv=128, R=0, r=r, B=B, H=H, S=S, steps=steps, seed=8000 + S + r,
                       symmetric=1)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    cut = S // 3
    cache.append(0, 0, _dev(k_host[:, :cut]), _dev(v_host[:, :cut]))
    cache.append(0, cut, _dev(k_host[:, cut:S]), _dev(v_host[:, cut:S]))
    _check_all_slices(cache, w, 0, S, k_host, v_host)
    q0 = synth.gen_q(w.seed, 0, range(w.batch), S - 1, w.n_q, w.d_head)
    _check_attention(cache, w, 0, S, k_host, v_host, q0, kvq.DECODE_MMA)
    with pytest.raises(kvq.KVQError):
        cache.attention(0, S, _dev(q0), softmax_scale(w), impl=kvq.DECODE_SIMT)
    for s in range(steps):
        T = S + s
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        out = cache.decode_step(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host),
                                softmax_scale(w)).cpu().numpy()
        if s == steps - 1:
            worst = 0.0
            for b in range(w.batch):
                for h in range(w.n_kv):
                    st = oracle_slice_state(k_host[b, :T + 1, h], v_host[b, :T + 1, h], cache)
                    ref = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
                    worst = max(worst, float(np.abs(out[b, h * w.gqa:(h + 1) * w.gqa] - ref).max()))
            assert worst <= ATOL, worst
    T = S + steps
    _check_all_slices(cache, w, 0, T, k_host, v_host)
    kd, vd = cache.dequantize(0, T)
    for b, h in {(0, 0), (w.batch - 1, w.n_kv - 1)}:
        st = oracle_slice_state(k_host[b, :T, h], v_host[b, :T, h], cache)
        kh, vh = oracle.dequantize_state_sym(st, d=128)
        assert np.array_equal(kd[b, h].cpu().numpy().view(np.uint32), kh.view(np.uint32))
        assert np.array_equal(vd[b, h].cpu().numpy().view(np.uint32), vh.view(np.uint32))


@pytest.mark.parametrize("k_out,r,B,H,S,steps", [
    (4, 4, 2, 2, 300, 4),     # small grid
    (1, 8, 2, 2, 257, 3),     # GQA 8, one entry per token
    (3, 4, 12, 4, 2100, 2),   # large grid
    (2, 2, 1, 3, 100, 2),     # GQA 2, two entries per token
])
def test_symmetric_with_outlier_isolation(k_out, r, B, H, S, steps):
    """Symmetric per-token int8 with k isolated key entries per token (dense-and-sparse):
    codes, scales and the sparse side list bit-exact after a chunked prefill and fused
    decode steps, attention (the sparse read path included) within 2e-3, and the
    dequantized keys bit-exact (the stored binary16 values at their channels)."""
    w = small_workload(bits=8, G=128, Gv=128, R=0, r=r, B=B, H=H, S=S, steps=steps, seed=9000 + S + k_out,
                       symmetric=1, k_outliers=k_out)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    cut = S // 2
    cache.append(0, 0, _dev(k_host[:, :cut]), _dev(v_host[:, :cut]))
    cache.append(0, cut, _dev(k_host[:, cut:S]), _dev(v_host[:, cut:S]))
    _check_all_slices(cache, w, 0, S, k_host, v_host)
    q0 = synth.gen_q(w.seed, 0, range(w.batch), S - 1, w.n_q, w.d_head)
    _check_attention(cache, w, 0, S, k_host, v_host, q0, kvq.DECODE_MMA)
    for s in range(steps):
        T = S + s
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        out = cache.decode_step(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host),
                                softmax_scale(w)).cpu().numpy()
        if s == steps - 1:
            worst = 0.0
            for b in range(w.batch):
                for h in range(w.n_kv):
                    st = oracle_slice_state(k_host[b, :T + 1, h], v_host[b, :T + 1, h], cache)
                    ref = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
                    worst = max(worst, float(np.abs(out[b, h * w.gqa:(h + 1) * w.gqa] - ref).max()))
            assert worst <= ATOL, worst
    T = S + steps
    _check_all_slices(cache, w, 0, T, k_host, v_host)
    kd, vd = cache.dequantize(0, T)
    for b, h in {(0, 0), (w.batch - 1, w.n_kv - 1)}:
        st = oracle_slice_state(k_host[b, :T, h], v_host[b, :T, h], cache)
        kh, vh = oracle.dequantize_state_sym(st, d=128)
        assert np.array_equal(kd[b, h].cpu().numpy().view(np.uint32), kh.view(np.uint32))
        assert np.array_equal(vd[b, h].cpu().numpy().view(np.uint32), vh.view(np.uint32))


def _adversarial_key_rows(rng):
    """Binary16 key rows that stress the outlier selection: the lower median of rows with
    signed zeros, constants, duplicates, two values, extremes and subnormals, and ties in
    |x - median| (broken towards the lower channel)."""
    d = 128
    rows = [np.zeros(d, np.float16)]                                    # all +0
    r = np.where(rng.random(d) < 0.5, np.float16(0.0), np.float16(-0.0)).astype(np.float16)
    r[17] = 5.0
    rows.append(r)                                                      # +0 / -0 mix, one entry away
    rows.append(np.full(d, 1.5, np.float16))                            # constant row
    rows.append((-np.abs(rng.standard_normal(d))).astype(np.float16))   # all negative
    rows.append(rng.integers(-1, 2, d).astype(np.float16))              # three values only
    r = rng.standard_normal(d).astype(np.float16)
    r[3], r[90] = 65504.0, -65504.0
    r[5], r[6], r[7] = np.float16(2.0 ** -24), -np.float16(2.0 ** -24), np.float16(2.0 ** -20)
    rows.append(r)                                                      # extremes and subnormals
    r = np.full(d, 2.0, np.float16)
    r[rng.permutation(d)[:64]] = -2.0
    rows.append(r)                                                      # two values, 64 each
    r = np.full(d, 0.25, np.float16)
    r[[10, 20, 30, 40, 50, 60]] = [3.0, -2.5, 3.0, -2.5, 3.0, -2.5]
    rows.append(r)                                                      # six entries at one distance
    r = rng.standard_normal(d).astype(np.float16)
    r[[100, 8, 64, 1]] = [-7.0, 7.0, -7.0, 7.0]
    rows.append(r)                                                      # four outliers of one magnitude
    return rows


def test_outlier_selection_on_adversarial_rows():
    """Outlier isolation on hand-built key rows (signed zeros, constant and two-valued
    rows, extremes, subnormals, distance ties), through the append kernel and through the
    fused decode step: codes, scales and the sparse side list bit-exact against the
    oracle, attention within 2e-3."""
    w = small_workload(bits=8, G=128, Gv=128, R=0, r=4, B=2, H=2, S=64, steps=2, seed=9100,
                       symmetric=1, k_outliers=4)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    k_host = np.array(k_host, dtype=np.float16)
    rows = _adversarial_key_rows(np.random.default_rng(9100))
    for i, row in enumerate(rows):
        k_host[0, i, 0] = row
        k_host[1, 20 + i, 1] = row[::-1]
    S = w.seq
    k_host[0, S, 0] = rows[1]  # the fused step quantizes these new rows
    k_host[1, S, 1] = rows[7]
    k_host[0, S + 1, 1] = rows[0]
    k_host[1, S + 1, 0] = rows[5]
    cache.append(0, 0, _dev(k_host[:, :S]), _dev(v_host[:, :S]))
    _check_all_slices(cache, w, 0, S, k_host, v_host)
    for s in range(w.steps):
        T = S + s
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        out = cache.decode_step(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host),
                                softmax_scale(w)).cpu().numpy()
        _check_all_slices(cache, w, 0, T + 1, k_host, v_host)
        for b in range(w.batch):
            for h in range(w.n_kv):
                st = oracle_slice_state(k_host[b, :T + 1, h], v_host[b, :T + 1, h], cache)
                ref = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
                err = float(np.abs(out[b, h * w.gqa:(h + 1) * w.gqa] - ref).max())
                assert err <= ATOL, (b, h, T + 1, err)


@pytest.mark.parametrize("kind", ["asym4", "int8", "sym8o4", "asym2-large", "sym8-large"])
def test_layer_interleaved_decode_with_early_prefetch(kind):
    """Decode steps that visit three layers in turn, as a model does: every launch after the
    first starts streaming its cache tiles before the previous layer's kernel has finished
    (KVQ_DECODE_EARLY_PREFETCH, set by the cache object). The asymmetric case fills a
    residual window during the steps (the two-launch path, which runs without the flag).
    The large-grid cases give the CTA that appends the new token several warps with
    early stages in flight while it appends. Every layer's cache state bit-exact and its
    attention within 2e-3 at every step, then an attention-only pass over the layers."""
    cfg = {
        "asym4": dict(bits=4, G=32, Gv=64, R=64, r=4, B=2, H=2, S=250, steps=8),
        "int8": dict(bits=8, G=128, Gv=128, R=0, r=4, B=1, H=4, S=500, steps=4),
        "sym8o4": dict(bits=8, G=128, Gv=128, R=0, r=4, B=2, H=2, S=300, steps=4, symmetric=1, k_outliers=4),
        "asym2-large": dict(bits=2, G=32, Gv=32, R=128, r=4, B=6, H=8, S=1500, steps=3),
        "sym8-large": dict(bits=8, G=128, Gv=128, R=0, r=4, B=6, H=8, S=1500, steps=3, symmetric=1),
    }[kind]
    w = small_workload(L=3, seed=9200 + len(kind), **cfg)
    cache = QuantizedKVCache.for_workload(w)
    host = [host_layer_inputs(w, layer, 0, w.max_seq) for layer in range(w.n_layers)]
    S = w.seq
    for layer in range(w.n_layers):
        cache.append(layer, 0, _dev(host[layer][0][:, :S]), _dev(host[layer][1][:, :S]))
    stream = torch.cuda.current_stream().cuda_stream
    flushed = False
    for s in range(w.steps):
        T = S + s
        for layer in range(w.n_layers):
            assert cache._early(stream, layer, None) == kvq.DECODE_EARLY_PREFETCH
            k_host, v_host = host[layer]
            flushed |= not w.symmetric and (T + 1) % max(w.residual, w.k_group) == 0
            q_host = synth.gen_q(w.seed, layer, range(w.batch), T, w.n_q, w.d_head)
            out = cache.decode_step(layer, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host),
                                    softmax_scale(w)).cpu().numpy()
            for b in range(w.batch):
                for h in range(w.n_kv):
                    st = oracle_slice_state(k_host[b, :T + 1, h], v_host[b, :T + 1, h], cache)
                    ref = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
                    err = float(np.abs(out[b, h * w.gqa:(h + 1) * w.gqa] - ref).max())
                    assert err <= ATOL, (kind, layer, b, h, T + 1, err)
    assert flushed == (kind == "asym4")
    T = S + w.steps
    for layer in range(w.n_layers):
        _check_all_slices(cache, w, layer, T, *host[layer])
    for layer in range(w.n_layers):
        q_host = synth.gen_q(w.seed, layer, range(w.batch), T - 1, w.n_q, w.d_head)
        _check_attention(cache, w, layer, T, *host[layer], q_host, kvq.DECODE_AUTO)


def _subnormals(n, sign_mix=True):
    """n binary16 subnormals k * 2^-24 with k in [1, 1023], mixed signs."""
    k = (np.arange(n) * 97 % 1023 + 1).astype(np.float64)
    s = np.where(np.arange(n) % 3 == 0, -1.0, 1.0) if sign_mix else 1.0
    return (s * k * 2.0**-24).astype(np.float16)


def _narrow(n, centre, step):
    """n values from {centre - step, centre, centre + step} (neighbouring binary16 values)."""
    return (centre + ((np.arange(n) % 3) - 1) * step).astype(np.float16)


def _edge_history(w):
    """Keys and values [B][T][H][d] of the seeded generator with planted edge groups:
    keys - a constant channel over a group (two signs), an all-zero group, narrow groups
    far from zero (around 7 and -1000: the widened scale), binary16 subnormals, and
    +-65504 in one channel (slice (0, 0) in the prompt; slice (1, 1) in the residual
    window that a decode step flushes); values - all-zero, constant, narrow-far-from-zero
    and subnormal groups in prompt rows and in rows appended by the fused step, and
    +-65504 groups in rows whose softmax weight is exactly 0 (their slice's attention is
    held by the +65504 key)."""
    k, v = host_layer_inputs(w, 0, 0, w.max_seq)
    k, v = np.array(k, np.float16), np.array(v, np.float16)
    S, Gv = w.seq, w.v_group
    g1 = slice(Gv, 2 * Gv) if w.d_head // Gv > 1 else slice(0, Gv)
    # keys of the prompt's quantized groups (G = 32)
    k[:, 0:32, :, 3] = 1.5
    k[:, 0:32, :, 4] = -0.75
    k[:, 32:64] = 0.0
    k[:, 64:96, :, 5] = _narrow(32, 7.0, 2.0**-8)[None, :, None]
    k[:, 64:96, :, 6] = _narrow(32, -1000.0, 0.5)[None, :, None]
    k[:, 96:128, :, 9] = _subnormals(32)[None, :, None]
    k[0, 96, 0, 7], k[0, 97, 0, 7] = 65504.0, -65504.0
    # keys of the residual window quantized by a decode step (tokens 128 .. 191)
    k[:, 128:160, :, 11] = 3.25
    k[:, 160:192, :, 12] = _narrow(32, 7.0, 2.0**-8)[None, :, None]
    k[:, 160:192, :, 14] = _subnormals(32)[None, :, None]
    k[1, 170, 1, 13], k[1, 180, 1, 13] = 65504.0, -65504.0
    # values: prompt rows 10..13 and fused-step rows S+1..S+4 in every slice
    for t in (10, S + 1):
        v[:, t, :, 0:Gv] = 0.0
    for t in (11, S + 2):
        v[:, t, :, g1] = -2.25
    for t in (12, S + 3):
        v[:, t, :, 0:Gv] = _narrow(Gv, 7.0, 2.0**-8)[None, None]
    for t in (13, S + 4):
        v[:, t, :, 0:Gv] = _subnormals(Gv)[None, None]
    ext = np.resize(np.array([65504.0, -65504.0, 0.0, 1.0], np.float16), Gv)
    v[0, 50, 0, 0:Gv] = ext
    v[0, S + 5, 0, 0:Gv] = ext
    v[1, 171, 1, 0:Gv] = ext
    return k, v


def _edge_queries(w, T):
    """Queries of the step at token T; query rows of slice (0, 0) read channel 7 and those of
    slice (1, 1) channel 13 with weight 1, so the planted +65504 keys hold their softmax."""
    q = np.array(synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head), np.float16)
    q[0, 0:w.gqa, 7] = 1.0
    q[1, w.gqa:2 * w.gqa, 13] = 1.0
    return q


@pytest.mark.parametrize("bits,Gv", [(8, 64), (4, 32), (2, 32)])
def test_asymmetric_edge_groups(bits, Gv):
    """Planted degenerate and extreme groups (see _edge_history) through the key-group and
    value-token append kernels (prompt), the fused decode step (new value rows, new key
    rows into the residual) and the key-group kernel of the step that fills the residual
    window: every byte of codes, metadata and residual bit-exact against the oracle,
    dequantized values bit-exact, attention within 2e-3 before and after the flush."""
    R = 64
    S = 2 * R + 20
    steps = R - 20 + 3  # the step at token 2R + R - 1 fills the window: tokens 128 .. 191 are quantized
    w = small_workload(bits=bits, G=32, Gv=Gv, R=R, r=4, B=2, H=2, S=S, steps=steps, seed=9300 + bits)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = _edge_history(w)
    cache.append(0, 0, _dev(k_host[:, :S]), _dev(v_host[:, :S]))
    _check_all_slices(cache, w, 0, S, k_host, v_host)
    flush_step = 3 * R - 1 - S
    for s in range(steps):
        T = S + s
        q_host = _edge_queries(w, T)
        out = cache.decode_step(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host),
                                softmax_scale(w)).cpu().numpy()
        if s not in (0, 5, 22, 23, flush_step, steps - 1):
            continue
        _check_all_slices(cache, w, 0, T + 1, k_host, v_host)
        for b in range(w.batch):
            for h in range(w.n_kv):
                st = oracle_slice_state(k_host[b, :T + 1, h], v_host[b, :T + 1, h], cache)
                ref = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
                err = float(np.abs(out[b, h * w.gqa:(h + 1) * w.gqa] - ref).max())
                assert err <= ATOL, (bits, b, h, T + 1, err)
    T = S + steps
    assert (T // R) * R == 3 * R  # the window of tokens 128 .. 191 was quantized
    kd, vd = cache.dequantize(0, T)
    for b in range(w.batch):
        for h in range(w.n_kv):
            st = oracle_slice_state(k_host[b, :T, h], v_host[b, :T, h], cache)
            kh, vh = oracle.dequantize_state(st, d=128, bits=bits, G=w.k_group, Gv=w.v_group, R=w.residual)
            assert np.array_equal(kd[b, h].cpu().numpy().view(np.uint32), kh.view(np.uint32)), (b, h)
            assert np.array_equal(vd[b, h].cpu().numpy().view(np.uint32), vh.view(np.uint32)), (b, h)
            if (b, h) == (0, 0):  # the +-65504 key group: widened to the full range, all other codes 0-ish
                assert np.abs(kh[96:98, 7]).min() > 20000


@pytest.mark.parametrize("B,H,S", [(2, 2, 700), (6, 8, 3000)])
def test_zero_wait_limit_reports_a_timeout(B, H, S):
    """KVQ_DECODE_ZERO_WAIT_LIMIT gives every bounded wait of the tensor-core kernel a limit
    of 0: each CTA gives up at its first wait, drains its copies and finishes (small grid:
    cluster merge; large grid: workspace merge). The launch returns KVQ_OK, the error word
    records the timeout and check_errors() raises; the next plain launch is correct and
    leaves the word clear (nothing faulted, the context stays usable)."""
    w = small_workload(bits=4, G=128, Gv=64, R=128, r=4, B=B, H=H, S=S, steps=1, seed=9400 + B)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    cache.append(0, 0, _dev(k_host[:, :S]), _dev(v_host[:, :S]))
    cache.check_errors()  # nothing recorded yet
    q_host = synth.gen_q(w.seed, 0, range(w.batch), S - 1, w.n_q, w.d_head)
    cache.attention(0, S, _dev(q_host), softmax_scale(w), flags=kvq.DECODE_ZERO_WAIT_LIMIT)
    with pytest.raises(kvq.KVQDeviceError) as e:
        cache.check_errors()
    assert e.value.word & kvq.DECODE_ERR_WAIT_TIMEOUT
    cache.check_errors()  # the read cleared it
    _check_attention(cache, w, 0, S, k_host, v_host, q_host, kvq.DECODE_AUTO)
    cache.check_errors()


@pytest.mark.parametrize("bits,v_bits,G,Gv,R,k_out,B,H", [
    (4, 0, 32, 64, 64, 2, 2, 2),     # small grid (cluster CTAs)
    (2, 0, 32, 32, 64, 4, 6, 8),     # large grid
    (8, 0, 128, 128, 128, 1, 2, 3),
    (8, 4, 64, 64, 128, 3, 6, 8),    # mixed widths, large grid
])
def test_per_channel_keys_with_isolated_entries(bits, v_bits, G, Gv, R, k_out, B, H):
    """Per-channel keys with k_out isolated entries per quantized key row: the key-group
    append kernel (prompt) and the step that fills the residual window split every row
    before forming its groups; the decode kernel adds the entries' score terms for
    quantized tokens. Codes, metadata, entry lists and residual bit-exact, dequantized keys
    bit-exact, attention within 2e-3 at every checked step, through the fused step."""
    R_eff = R
    S = 2 * R_eff + 10
    steps = R_eff - 10 + 3
    w = small_workload(bits=bits, v_bits=v_bits, G=G, Gv=Gv, R=R, r=4, B=B, H=H, S=S, steps=steps, n_out=4,
                       seed=9500 + bits + k_out, k_outliers=k_out)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    cache.append(0, 0, _dev(k_host[:, :S]), _dev(v_host[:, :S]))
    _check_all_slices(cache, w, 0, S, k_host, v_host)
    flush_step = 3 * R_eff - 1 - S
    for s in range(steps):
        T = S + s
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        out = cache.decode_step(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host),
                                softmax_scale(w)).cpu().numpy()
        if s not in (0, flush_step - 1, flush_step, steps - 1):
            continue
        _check_all_slices(cache, w, 0, T + 1, k_host, v_host)
        for b in range(w.batch):
            for h in range(w.n_kv):
                st = oracle_slice_state(k_host[b, :T + 1, h], v_host[b, :T + 1, h], cache)
                ref = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
                err = float(np.abs(out[b, h * w.gqa:(h + 1) * w.gqa] - ref).max())
                assert err <= ATOL, (b, h, T + 1, err)
    T = S + steps
    kd, vd = cache.dequantize(0, T)
    for b in range(w.batch):
        for h in range(w.n_kv):
            st = oracle_slice_state(k_host[b, :T, h], v_host[b, :T, h], cache)
            assert st.k_sparse is not None and st.k_sparse.shape[1] == k_out
            kh, vh = oracle.dequantize_state(st, d=128, bits=bits, G=G, Gv=Gv, R=R, v_bits=v_bits)
            assert np.array_equal(kd[b, h].cpu().numpy().view(np.uint32), kh.view(np.uint32)), (b, h)
            assert np.array_equal(vd[b, h].cpu().numpy().view(np.uint32), vh.view(np.uint32)), (b, h)


def test_per_channel_key_outliers_on_adversarial_rows():
    """The key-group kernel's row split on hand-built key rows (signed zeros, constant and
    two-valued rows, extremes, subnormals, distance ties) in the prompt and in the residual
    window a decode step flushes: state bit-exact, attention within 2e-3."""
    w = small_workload(bits=4, G=32, Gv=64, R=64, r=4, B=2, H=2, S=128 + 10, steps=58, seed=9600, k_outliers=4)
    cache = QuantizedKVCache.for_workload(w)
    k_host, v_host = host_layer_inputs(w, 0, 0, w.max_seq)
    k_host = np.array(k_host, dtype=np.float16)
    rows = _adversarial_key_rows(np.random.default_rng(9600))
    for i, row in enumerate(rows):
        k_host[0, 3 + i, 0] = row            # prompt rows
        k_host[1, 140 + i, 1] = row[::-1]    # rows flushed by a decode step
    S = w.seq
    cache.append(0, 0, _dev(k_host[:, :S]), _dev(v_host[:, :S]))
    _check_all_slices(cache, w, 0, S, k_host, v_host)
    for s in range(w.steps):
        T = S + s
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        out = cache.decode_step(0, T, _dev(k_host[:, T:T + 1]), _dev(v_host[:, T:T + 1]), _dev(q_host),
                                softmax_scale(w)).cpu().numpy()
        if T + 1 not in (S + 1, 192, S + w.steps):
            continue
        _check_all_slices(cache, w, 0, T + 1, k_host, v_host)
        for b in range(w.batch):
            for h in range(w.n_kv):
                st = oracle_slice_state(k_host[b, :T + 1, h], v_host[b, :T + 1, h], cache)
                ref = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, softmax_scale(w))
                err = float(np.abs(out[b, h * w.gqa:(h + 1) * w.gqa] - ref).max())
                assert err <= ATOL, (b, h, T + 1, err)
