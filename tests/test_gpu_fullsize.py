"""Full-size parity: every benchmark workload at its real shape, in the launch
configuration the benchmark times, checked on sampled (batch row, kv head) slices of
the first and last layer (bit-exact cache state) and on the attention outputs of those
slices at the first and last decode step (max-abs 2e-3)."""

import zlib

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from kvq_testlib import ATOL, assert_slice_equal, gpu_slice_state, oracle_attention, oracle_slice_state  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from bit_kv_cache_09_gb300.cache import QuantizedKVCache  # noqa: E402
from synth.device import DeviceGenerator  # noqa: E402

FULL = ["llama8b-int8", "kivi-int4", "kivi-int2", "kivi-k8v4", "llama8b-sym8", "sym8-b16", "sym8o4-b16", "long-int4-16k", "long-int4-32k", "long-int4-64k"]


def _samples(w, rng):
    picks = {(0, 0), (w.batch - 1, w.n_kv - 1)}
    picks.add((int(rng.integers(w.batch)), int(rng.integers(w.n_kv))))
    return sorted(picks)


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name):
    w = synth.WORKLOADS[name]
    rng = np.random.default_rng(zlib.crc32(name.encode()))
    cache = QuantizedKVCache.for_workload(w)
    gen = DeviceGenerator(w)
    S, L = w.seq, w.n_layers
    chunk = max(128, min(S, (1 << 28) // (w.batch * w.n_kv * w.d_head * 2) // 128 * 128))
    worst = 0.0
    for layer in (0, L - 1):
        t = 0
        while t < S:  # prefill exactly as the benchmark does
            n = min(chunk, S - t)
            k, v = gen.kv(layer, t, n)
            cache.append(layer, t, k, v)
            t += n
        samples = _samples(w, rng)
        hist = {(b, h): (synth.k_slice(w, layer, b, h, range(w.max_seq)), synth.v_slice(w, layer, b, h, range(w.max_seq)))
                for b, h in samples}
        for b, h in samples:
            kh, vh = hist[(b, h)]
            st = oracle_slice_state(kh[:S], vh[:S], cache)
            assert_slice_equal(gpu_slice_state(cache, layer, b, h, S), st, f"{name} l={layer} b={b} h={h} prefill")
        for step in range(w.steps):
            T = S + step
            k, v = gen.kv(layer, T, 1)
            cache.append(layer, T, k, v)
            if step not in (0, w.steps - 1):
                continue
            q = gen.q(layer, T)
            out = cache.attention(layer, T + 1, q, w.softmax_scale).cpu().numpy()
            qh = q.cpu().numpy()
            for b, h in samples:
                kh, vh = hist[(b, h)]
                st = oracle_slice_state(kh[:T + 1], vh[:T + 1], cache)
                assert_slice_equal(gpu_slice_state(cache, layer, b, h, T + 1), st, f"{name} l={layer} b={b} h={h} T={T + 1}")
                ref = oracle_attention(st, qh[b, h * w.gqa:(h + 1) * w.gqa], cache, w.softmax_scale)
                err = float(np.abs(out[b, h * w.gqa:(h + 1) * w.gqa] - ref).max())
                worst = max(worst, err)
                assert err <= ATOL, (name, layer, b, h, T + 1, err)
    # layers in between were never written
    kc = cache.buffer("k_codes")
    per_layer = kc.numel() // L
    if L > 2:
        assert not kc[per_layer: 2 * per_layer].any()
    print(f"{name}: worst attention error {worst:.2e}")


def test_full_size_dequantize_sampled():
    w = synth.WORKLOADS["kivi-int2"]
    cache = QuantizedKVCache.for_workload(w, n_layers=1)
    gen = DeviceGenerator(w)
    T = w.seq + 5
    k, v = gen.kv(0, 0, T)
    cache.append(0, 0, k, v)
    kd, vd = cache.dequantize(0, T)
    for b, h in [(0, 0), (w.batch - 1, 3), (17, w.n_kv - 1)]:
        kh = synth.k_slice(w, 0, b, h, range(T))
        vh = synth.v_slice(w, 0, b, h, range(T))
        st = oracle_slice_state(kh, vh, cache)
        ko, vo = oracle.dequantize_state(st, d=128, bits=w.bits, G=w.k_group, Gv=w.v_group, R=w.residual)
        assert np.array_equal(kd[b, h].cpu().numpy().view(np.uint32), ko.view(np.uint32))
        assert np.array_equal(vd[b, h].cpu().numpy().view(np.uint32), vo.view(np.uint32))
