"""Full-size parity: every benchmark workload at its real shape, in the launch
configuration the benchmark times (prefill in the benchmark's chunks, then decode steps
through the fused kvq_decode_step launch, the first and the last layer in turn so that
every launch after the first streams its first tiles early). Every (batch row, kv head)
slice of both layers is checked: the packed cache state after the last step bit-exact,
and the attention outputs of the first and the last decode step within 2e-3. The oracle
runs in a spawned process pool (single-threaded per slice)."""

import multiprocessing as mp
import os

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
import synth  # noqa: E402
from kvq_testlib import ATOL, assert_slice_equal, gpu_slice_state, oracle_slice_job, oracle_slice_state  # noqa: E402

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from bit_kv_cache_09_gb300 import kvq  # noqa: E402
from bit_kv_cache_09_gb300.cache import QuantizedKVCache  # noqa: E402
from synth.device import DeviceGenerator  # noqa: E402

FULL = ["llama8b-int8", "kivi-int4", "kivi-int2", "kivi-k8v4", "llama8b-sym8", "sym8-b16", "sym8o4-b16",
        "kivi-int4o4", "long-int4-16k", "long-int4-32k", "long-int4-64k"]


@pytest.fixture(scope="module")
def pool():
    # spawned workers (never forked from a process that holds a CUDA context)
    ctx = mp.get_context("spawn")
    n = max(1, min(16, (os.cpu_count() or 2) - 1))
    with ctx.Pool(n) as p:
        yield p


@pytest.mark.parametrize("name", FULL)
def test_full_size_workload(name, pool):
    w = synth.WORKLOADS[name]
    cache = QuantizedKVCache.for_workload(w)
    gen = DeviceGenerator(w)
    S, L = w.seq, w.n_layers
    layers = (0, L - 1)
    chunk = max(128, min(S, (1 << 28) // (w.batch * w.n_kv * w.d_head * 2) // 128 * 128))
    for layer in layers:
        t = 0
        while t < S:  # prefill exactly as the benchmark does
            n = min(chunk, S - t)
            k, v = gen.kv(layer, t, n)
            cache.append(layer, t, k, v)
            t += n
    stream = torch.cuda.current_stream().cuda_stream
    first, last = S + 1, S + w.steps
    outs, qs = {}, {}
    for step in range(w.steps):
        T = S + step
        for layer in layers:
            # the previous launch on the stream wrote the other layer: early prefetch is on
            assert L == 1 or step == 0 and layer == 0 or cache._early(stream, layer, None) == kvq.DECODE_EARLY_PREFETCH
            k, v = gen.kv(layer, T, 1)
            q = gen.q(layer, T)
            out = cache.decode_step(layer, T, k, v, q, w.softmax_scale)
            if T + 1 in (first, last):
                outs[(layer, T + 1)] = out.cpu().numpy()
                qs[(layer, T + 1)] = q.cpu().numpy()
    torch.cuda.synchronize()
    jobs = []
    for layer in layers:
        for b in range(w.batch):
            for h in range(w.n_kv):
                jobs.append({"w": w, "layer": layer, "b": b, "h": h, "Ts": sorted({first, last}),
                             "q": {T: qs[(layer, T)][b, h * w.gqa:(h + 1) * w.gqa] for T in (first, last)}})
    worst, n_slices = 0.0, 0
    for res in pool.imap_unordered(oracle_slice_job, jobs, chunksize=4):
        layer, b, h = res["key"]
        assert_slice_equal(gpu_slice_state(cache, layer, b, h, last), res["state"], f"{name} l={layer} b={b} h={h}")
        for T, ref in res["att"].items():
            err = float(np.abs(outs[(layer, T)][b, h * w.gqa:(h + 1) * w.gqa] - ref).max())
            worst = max(worst, err)
            assert err <= ATOL, (name, layer, b, h, T, err)
        n_slices += 1
    assert n_slices == len(layers) * w.batch * w.n_kv
    # layers in between were never written
    kc = cache.buffer("k_codes")
    per_layer = kc.numel() // L
    if L > 2:
        assert not kc[per_layer: 2 * per_layer].any()
    print(f"{name}: {n_slices} slices, worst attention error {worst:.2e}")


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
