"""The allocation-free decode entry point against the regular one.

kvq_decode_attention_noalloc serves callers that cannot allocate device memory at
the call site: it keeps the split-K scratch in a static device array instead of a
caller workspace. Two calls in a row (the array keeps the first call's contents)
must give the regular entry point's outputs within the attention tolerance.
This file is collected last on purpose.
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

ATOL = 2e-3


def test_noalloc_matches_workspace_entry_point_twice():
    kvq_build.build()
    w = synth.Workload("noalloc", 1, 2, 4, 128, 3, 1500, 2, 4, 128, 64, 128, 4, 20, 31337)
    cache = QuantizedKVCache.for_workload(w)
    toks = np.arange(w.max_seq)
    k = synth.gen_k(w.seed, 0, range(w.batch), toks, w.n_kv, w.d_head, w.n_out, w.gain)
    v = synth.gen_v(w.seed, 0, range(w.batch), toks, w.n_kv, w.d_head)
    kd, vd = torch.from_numpy(k).cuda(), torch.from_numpy(v).cuda()
    cache.append(0, 0, kd[:, :w.seq].contiguous(), vd[:, :w.seq].contiguous())
    stream = torch.cuda.current_stream().cuda_stream
    for step in range(2):
        T = w.seq + step
        cache.append(0, T, kd[:, T:T + 1].contiguous(), vd[:, T:T + 1].contiguous())
        q = torch.from_numpy(synth.gen_q(w.seed, 0, range(w.batch), T, w.n_q, w.d_head)).cuda()
        assert kvq.kvq_decode_num_splits(cache.cfg, T + 1) > 1  # the scratch is really used
        ref = cache.attention(0, T + 1, q, w.softmax_scale)
        out = torch.full_like(ref, float("nan"))
        kvq.kvq_decode_attention_noalloc(cache.cfg, cache.bufs, 0, T + 1, q.data_ptr(), w.softmax_scale,
                                         out.data_ptr(), stream)
        torch.cuda.synchronize()
        assert torch.isfinite(out).all()
        assert (out - ref).abs().max().item() <= ATOL


def test_noalloc_rejects_configs_beyond_its_scratch():
    cfg = kvq.make_config(n_layers=1, batch=4095, n_kv_heads=8, gqa_ratio=8, d_head=128, max_seq_len=1 << 16, bits=4,
                          k_group=128, v_group=128, residual_len=128)
    assert kvq.kvq_decode_workspace_size(cfg, 1 << 16) > 16 << 20
    bufs = kvq.make_buffers([256] * 5)
    with pytest.raises(kvq.KVQError) as e:
        kvq.kvq_decode_attention_noalloc(cfg, bufs, 0, 1 << 16, 256, 0.1, 256, 0)
    assert e.value.status == 4  # KVQ_ERR_WORKSPACE, before any launch
