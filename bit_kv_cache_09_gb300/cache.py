"""Device-memory harness around the C ABI: PyTorch allocates, libkvq computes.

``QuantizedKVCache`` owns the five cache buffers and a decode workspace as torch
tensors and forwards every call to the ``kvq_*`` entry points with the tensors'
device addresses and the current CUDA stream. No arithmetic of the path happens
here.

Decode launches pass ``KVQ_DECODE_EARLY_PREFETCH`` (their first cache tiles stream in
while the previous kernel of the stream finishes) unless this object's previous launch
on the same stream wrote the same layer. Kernels that write the cache buffers outside
this object (through ``buffer()``) must therefore not directly precede a decode launch
on the same stream; pass ``early=False`` after them.
"""

from __future__ import annotations

import torch

from . import kvq


class QuantizedKVCache:
    def __init__(self, *, n_layers, batch, n_kv_heads, gqa_ratio, d_head, max_seq_len, bits, k_group, v_group,
                 residual_len, v_bits=0, symmetric=0, k_outliers=0, device="cuda"):
        self.cfg = kvq.make_config(n_layers=n_layers, batch=batch, n_kv_heads=n_kv_heads, gqa_ratio=gqa_ratio,
                                   d_head=d_head, max_seq_len=max_seq_len, bits=bits, k_group=k_group,
                                   v_group=v_group, residual_len=residual_len, v_bits=v_bits, symmetric=symmetric,
                                   k_outliers=k_outliers)
        self.device = torch.device(device)
        sizes = kvq.kvq_buffer_sizes(self.cfg)
        # byte buffers, zero-filled as the ABI requires; torch allocations are 256-byte aligned
        self.buffers = [torch.zeros(max(s, 16), dtype=torch.uint8, device=self.device) for s in sizes]
        self.bufs = kvq.make_buffers([b.data_ptr() for b in self.buffers])
        self.ws = torch.zeros(max(kvq.kvq_decode_workspace_size(self.cfg, max_seq_len), 16), dtype=torch.uint8,
                              device=self.device)
        self.n_q = n_kv_heads * gqa_ratio
        self._last = None  # (stream, layer, wrote) of this object's previous launch

    @classmethod
    def for_workload(cls, w, *, n_layers=None, device="cuda"):
        return cls(n_layers=n_layers or w.n_layers, batch=w.batch, n_kv_heads=w.n_kv, gqa_ratio=w.gqa,
                   d_head=w.d_head, max_seq_len=w.max_seq, bits=w.bits, k_group=w.k_group, v_group=w.v_group,
                   residual_len=w.residual, v_bits=w.v_bits, symmetric=w.symmetric, k_outliers=w.k_outliers,
                   device=device)

    @staticmethod
    def _stream() -> int:
        return torch.cuda.current_stream().cuda_stream

    def buffer(self, name: str) -> torch.Tensor:
        return self.buffers[kvq.BUFFER_NAMES.index(name)]

    def _early(self, stream: int, layer: int, early) -> int:
        """Flag bits of a decode launch of `layer` on `stream` (see the module docstring)."""
        if early is None:
            early = not (self._last is not None and self._last[0] == stream and self._last[1] == layer
                         and self._last[2])
        return kvq.DECODE_EARLY_PREFETCH if early else 0

    def check_errors(self) -> None:
        """Raise KVQDeviceError if a decode launch since the last check recorded a
        device-side error (a bounded wait that ran out); clears the word. Synchronizes
        the current stream."""
        word = kvq.kvq_decode_error(self.ws.data_ptr(), self.ws.numel(), self._stream())
        if word:
            raise kvq.KVQDeviceError(word)

    def append(self, layer: int, s_cur: int, k: torch.Tensor, v: torch.Tensor) -> None:
        """k, v: [batch][n_new][n_kv_heads][d_head] float16 on the device."""
        assert k.dtype == torch.float16 and v.dtype == torch.float16 and k.is_contiguous() and v.is_contiguous()
        assert k.shape == v.shape and k.dim() == 4
        stream = self._stream()
        kvq.kvq_quantize_append(self.cfg, self.bufs, layer, s_cur, k.shape[1], k.data_ptr(), v.data_ptr(), stream)
        self._last = (stream, layer, True)

    def dequantize(self, layer: int, s_cur: int):
        c = self.cfg
        k_out = torch.empty((c.batch, c.n_kv_heads, s_cur, c.d_head), dtype=torch.float32, device=self.device)
        v_out = torch.empty_like(k_out)
        stream = self._stream()
        kvq.kvq_dequantize(self.cfg, self.bufs, layer, s_cur, k_out.data_ptr(), v_out.data_ptr(), stream)
        self._last = (stream, layer, False)
        return k_out, v_out

    def attention(self, layer: int, s_cur: int, q: torch.Tensor, softmax_scale: float, out: torch.Tensor = None,
                  impl: int = kvq.DECODE_AUTO, early=None, flags: int = 0) -> torch.Tensor:
        """q: [batch][n_q][d_head] float16; returns out [batch][n_q][d_head] float32.
        flags: extra kvq_decode_attention_ex flag bits (KVQ_DECODE_ZERO_WAIT_LIMIT)."""
        assert q.dtype == torch.float16 and q.is_contiguous()
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=self.device)
        stream = self._stream()
        if impl == kvq.DECODE_AUTO:
            kvq.kvq_decode_attention_ex(self.cfg, self.bufs, layer, s_cur, q.data_ptr(), softmax_scale,
                                        out.data_ptr(), self.ws.data_ptr(), self.ws.numel(), stream,
                                        self._early(stream, layer, early) | flags)
        else:
            kvq.kvq_decode_attention_impl(self.cfg, self.bufs, layer, s_cur, q.data_ptr(), softmax_scale,
                                          out.data_ptr(), self.ws.data_ptr(), self.ws.numel(), stream, impl)
        self._last = (stream, layer, False)
        return out

    def decode_step(self, layer: int, s_cur: int, k: torch.Tensor, v: torch.Tensor, q: torch.Tensor,
                    softmax_scale: float, out: torch.Tensor = None, early=None) -> torch.Tensor:
        """Append one token ([batch][1][n_kv][d] float16) and attend over s_cur + 1 tokens."""
        assert k.dtype == torch.float16 and v.dtype == torch.float16 and q.dtype == torch.float16
        assert k.is_contiguous() and v.is_contiguous() and q.is_contiguous() and k.shape[1] == 1
        if out is None:
            out = torch.empty(q.shape, dtype=torch.float32, device=self.device)
        stream = self._stream()
        kvq.kvq_decode_step_ex(self.cfg, self.bufs, layer, s_cur, k.data_ptr(), v.data_ptr(), q.data_ptr(),
                               softmax_scale, out.data_ptr(), self.ws.data_ptr(), self.ws.numel(), stream,
                               self._early(stream, layer, early))
        self._last = (stream, layer, True)
        return out
