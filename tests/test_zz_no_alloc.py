"""The allocation-free decode entry point.

kvq_decode_attention_noalloc serves callers that cannot allocate device memory where
they call it (a host framework whose allocator owns all device memory, or a decode loop
that cannot take an allocation's implicit device synchronisation): its split-K scratch is
a static device array of the library instead of a caller workspace. The shape here has
enough (batch row, kv head) pairs and a split count outside {2, 4, 8}, so every pair's
partials go through that array and the last CTA of each pair merges them from there.
Two calls in a row (the array keeps the first call's contents) must match the oracle
within 2e-3 and the workspace entry point's outputs exactly. This file is collected
last on purpose.
"""

import numpy as np
import pytest

torch = pytest.importorskip("torch")

pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import synth  # noqa: E402
from bit_kv_cache_09_gb300 import build as kvq_build  # noqa: E402
from bit_kv_cache_09_gb300 import kvq  # noqa: E402
from bit_kv_cache_09_gb300.cache import QuantizedKVCache  # noqa: E402
from kvq_testlib import ATOL, oracle_attention, oracle_slice_state  # noqa: E402


def test_noalloc_partials_go_through_the_static_array_twice():
    kvq_build.build()
    B, H = 6, 8  # 48 pairs: a large grid, merged through the workspace unless 2, 4 or 8 splits
    cfg0 = kvq.make_config(n_layers=1, batch=B, n_kv_heads=H, gqa_ratio=4, d_head=128, max_seq_len=6100, bits=4,
                           k_group=128, v_group=64, residual_len=128)
    # a prompt length whose split plan merges through the workspace (n_split not 1, 2, 4, 8)
    S = next(s for s in range(2998, 6000, 61)
             if all(kvq.kvq_decode_num_splits(cfg0, T) not in (1, 2, 4, 8) for T in (s + 1, s + 2)))
    w = synth.Workload("noalloc", 1, H, 4, 128, B, S, 2, 4, 128, 64, 128, 4, 20, 31337)
    cache = QuantizedKVCache.for_workload(w)
    toks = np.arange(w.max_seq)
    k = synth.gen_k(w.seed, 0, range(w.batch), toks, w.n_kv, w.d_head, w.n_out, w.gain)
    v = synth.gen_v(w.seed, 0, range(w.batch), toks, w.n_kv, w.d_head)
    kd, vd = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    cache.append(0, 0, kd[:, :S].contiguous(), vd[:, :S].contiguous())
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(2):
        T = S + step
        cache.append(0, T, kd[:, T:T + 1].contiguous(), vd[:, T:T + 1].contiguous())
        n_split = kvq.kvq_decode_num_splits(cache.cfg, T + 1)
        assert n_split > 2 and n_split not in (4, 8)  # partials and tickets live in the static array
        q_host = synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)
        q = torch.from_numpy(q_host).cuda()
        ref = cache.attention(0, T + 1, q, w.softmax_scale)
        out = torch.full_like(ref, float("nan"))
        kvq.kvq_decode_attention_noalloc(cache.cfg, cache.bufs, 0, T + 1, q.data_ptr(), w.softmax_scale,
                                         out.data_ptr(), stream)
        assert kvq.kvq_decode_noalloc_error(stream) == 0  # synchronizes
        assert torch.equal(out, ref)  # the same kernels and plan as the workspace entry point
        got = out.cpu().numpy()
        for b in range(B):
            for h in range(H):
                st = oracle_slice_state(k[b, :T + 1, h], v[b, :T + 1, h], cache)
                exp = oracle_attention(st, q_host[b, h * w.gqa:(h + 1) * w.gqa], cache, w.softmax_scale)
                err = float(np.abs(got[b, h * w.gqa:(h + 1) * w.gqa] - exp).max())
                assert err <= ATOL, (step, b, h, err)


def test_noalloc_rejects_configs_beyond_its_scratch():
    cfg = kvq.make_config(n_layers=1, batch=4095, n_kv_heads=8, gqa_ratio=8, d_head=128, max_seq_len=1 << 16, bits=4,
                          k_group=128, v_group=128, residual_len=128)
    assert kvq.kvq_decode_workspace_size(cfg, 1 << 16) > 16 << 20
    bufs = kvq.make_buffers([256] * 5)
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_decode_attention_noalloc(cfg, bufs, 0, 1 << 16, 256, 0.1, 256, 0)
    assert e.value.status == 4  # KVQ_ERR_WORKSPACE, before any launch


def test_noalloc_checks_arguments_before_touching_its_array():
    """A call with a bad argument is rejected on the host (it writes nothing to the shared
    array, which another stream's decode may be using)."""
    cfg = kvq.make_config(n_layers=1, batch=2, n_kv_heads=2, gqa_ratio=4, d_head=128, max_seq_len=1000, bits=4,
                          k_group=128, v_group=64, residual_len=128)
    good = kvq.make_buffers([256] * 5)
    cases = [(kvq.make_buffers([256, 256, 0, 256, 256]), 0, 500, 256, 0.1, 1),  # null buffer
             (good, 1, 500, 256, 0.1, 1),                                      # layer out of range
             (good, 0, 500, 260, 0.1, 1),                                      # misaligned query
             (good, 0, 1001, 256, 0.1, 3),                                     # beyond capacity
             (good, 0, 500, 256, float("inf"), 1)]                             # bad softmax scale
    for bufs, layer, s, qp, scale, status in cases:
        with pytest.raises(kvq.KVQError) as e:
            kvq.kvq_decode_attention_noalloc(cfg, bufs, layer, s, qp, scale, 256, 0)
        assert e.value.status == status
