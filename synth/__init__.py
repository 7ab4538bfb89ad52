"""Seeded synthetic K / V / query generator and the workload table.

This module holds none of the quantization or attention arithmetic. It is the
one piece shared by the oracle side (tests) and the CUDA side (tests, bench):
the host implementation below (numpy) and the device implementation in
``synth_gen.cu`` follow the same published counter-based definition, so any
slice of any workload can be generated on either side, bit for bit.

Definition
----------
* ``mix64`` is the splitmix64 finaliser (Steele, Lea, Flood, "Fast splittable
  pseudorandom number generators", OOPSLA 2014):
  ``x ^= x >> 30; x *= 0xbf58476d1ce4e5b9; x ^= x >> 27; x *= 0x94d049bb133111eb; x ^= x >> 31``.
* Counter of one element: ``(stream << 60) | (layer << 52) | (head << 44) |
  (channel << 36) | (batch << 24) | token`` (stream 0 = K, 1 = V, 2 = query,
  3 = outlier-channel pick). Limits: layer, head, channel < 256, batch < 4096,
  token < 2**24.
* ``base = mix64((seed * 0x9E3779B97F4A7C15) ^ counter)``; three words
  ``w_k = mix64(base + k * 0x9E3779B97F4A7C15)`` for k = 1, 2, 3 give twelve
  16-bit uniforms u_i; ``m = sum(u_i) - 6 * 65536`` and ``z = m / 65536`` (an
  Irwin–Hall approximation of N(0, 1); z is exact in binary32).
* K, normal channel: binary16(z). K, outlier channel:
  binary16(binary32(a * m + shift * 65536) * 2**-16) — the integer is converted
  to binary32 with round-to-nearest-even, then scaled exactly.
  V: binary16(z / 2). Query: binary16(z). Every binary16 conversion rounds to
  nearest-even.
* Outlier channels of (layer, kv head): draw ``mix64((seed * golden) ^
  counter(3, layer, head, 0, 0, k)) % d_head`` for k = 0, 1, ... and keep the
  first ``n_out`` distinct values. They are shared by every batch row and token.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

GOLDEN = 0x9E3779B97F4A7C15
M1 = 0xBF58476D1CE4E5B9
M2 = 0x94D049BB133111EB
STREAM_K, STREAM_V, STREAM_Q, STREAM_PICK = 0, 1, 2, 3


def mix64(x: np.ndarray) -> np.ndarray:
    """splitmix64 finaliser on a uint64 array (wrapping arithmetic)."""
    x = np.asarray(x, dtype=np.uint64).copy()
    with np.errstate(over="ignore"):
        x ^= x >> np.uint64(30)
        x *= np.uint64(M1)
        x ^= x >> np.uint64(27)
        x *= np.uint64(M2)
        x ^= x >> np.uint64(31)
    return x


def counter(stream, layer, head, channel, batch, token) -> np.ndarray:
    u = np.uint64
    return ((u(stream) << u(60)) | (np.asarray(layer, np.uint64) << u(52)) | (np.asarray(head, np.uint64) << u(44))
            | (np.asarray(channel, np.uint64) << u(36)) | (np.asarray(batch, np.uint64) << u(24))
            | np.asarray(token, np.uint64))


def normal_m(seed: int, ctr: np.ndarray) -> np.ndarray:
    """Integer m = sum of twelve 16-bit uniforms - 6*65536 (int64), per counter."""
    with np.errstate(over="ignore"):
        base = mix64((np.uint64((seed * GOLDEN) & (2**64 - 1))) ^ np.asarray(ctr, np.uint64))
        total = np.zeros(base.shape, np.int64)
        for k in (1, 2, 3):
            w = mix64(base + np.uint64((k * GOLDEN) & (2**64 - 1)))
            for s in (0, 16, 32, 48):
                total += ((w >> np.uint64(s)) & np.uint64(0xFFFF)).astype(np.int64)
    return total - 6 * 65536


def outlier_channels(seed: int, layer: int, head: int, n_out: int, d: int = 128) -> list[int]:
    out: list[int] = []
    k = 0
    while len(out) < n_out:
        with np.errstate(over="ignore"):
            x = mix64(np.uint64((seed * GOLDEN) & (2**64 - 1)) ^ counter(STREAM_PICK, layer, head, 0, 0, k))
        c = int(x % np.uint64(d))
        if c not in out:
            out.append(c)
        k += 1
    return out


def outlier_mask_words(seed: int, layer: int, n_kv: int, n_out: int, d: int = 128) -> np.ndarray:
    """[n_kv][d/64] uint64 bit masks of the outlier channels of one layer."""
    words = np.zeros((n_kv, (d + 63) // 64), np.uint64)
    for h in range(n_kv):
        for c in outlier_channels(seed, layer, h, n_out, d):
            words[h, c // 64] |= np.uint64(1) << np.uint64(c % 64)
    return words


def _to_f16(x32: np.ndarray) -> np.ndarray:
    return x32.astype(np.float32).astype(np.float16)


def gen_k(seed, layer, batches, tokens, n_kv, d, n_out, a, shift=5.0, heads=None) -> np.ndarray:
    """Keys [len(batches)][len(tokens)][len(heads)][d] binary16 (heads default: all n_kv)."""
    heads = np.arange(n_kv, dtype=np.int64) if heads is None else np.asarray(heads, np.int64)
    b = np.asarray(batches, np.int64)[:, None, None, None]
    t = np.asarray(tokens, np.int64)[None, :, None, None]
    h = heads[None, None, :, None]
    c = np.arange(d, dtype=np.int64)[None, None, None, :]
    m = normal_m(seed, counter(STREAM_K, layer, h, c, b, t))
    out = m.astype(np.float32) * np.float32(2.0**-16)  # exact
    if n_out > 0:
        mask = np.zeros((len(heads), d), bool)
        for j, hh in enumerate(heads):
            mask[j, outlier_channels(seed, layer, int(hh), n_out, d)] = True
        mask = np.broadcast_to(mask[None, None], m.shape)
        ai = int(a)
        assert ai == a, "outlier gain must be an integer"
        big = (m * ai + int(round(shift * 65536))).astype(np.float64).astype(np.float32) * np.float32(2.0**-16)
        out = np.where(mask, big, out)
    return _to_f16(out)


def gen_v(seed, layer, batches, tokens, n_kv, d, heads=None) -> np.ndarray:
    """Values [len(batches)][len(tokens)][len(heads)][d] binary16, sigma 0.5."""
    heads = np.arange(n_kv, dtype=np.int64) if heads is None else np.asarray(heads, np.int64)
    b = np.asarray(batches, np.int64)[:, None, None, None]
    t = np.asarray(tokens, np.int64)[None, :, None, None]
    h = heads[None, None, :, None]
    c = np.arange(d, dtype=np.int64)[None, None, None, :]
    m = normal_m(seed, counter(STREAM_V, layer, h, c, b, t))
    return _to_f16(m.astype(np.float32) * np.float32(2.0**-17))


def gen_q(seed, layer, batches, step_token, n_q, d) -> np.ndarray:
    """Queries [len(batches)][n_q][d] binary16 for the decode step at token index ``step_token``."""
    b = np.asarray(batches, np.int64)[:, None, None]
    i = np.arange(n_q, dtype=np.int64)[None, :, None]
    c = np.arange(d, dtype=np.int64)[None, None, :]
    m = normal_m(seed, counter(STREAM_Q, layer, i, c, b, step_token))
    return _to_f16(m.astype(np.float32) * np.float32(2.0**-16))


# ----------------------------------------------------------------------------- workloads
@dataclass(frozen=True)
class Workload:
    """One synthetic workload: cache shape, quantizer settings and generator parameters."""

    name: str
    n_layers: int
    n_kv: int
    gqa: int
    d_head: int
    batch: int
    seq: int  # prompt tokens quantized by the prefill
    steps: int  # decode steps appended after the prompt
    bits: int
    k_group: int
    v_group: int
    residual: int  # 0 => residual capacity equals k_group
    n_out: int
    gain: int
    seed: int
    shift: float = 5.0
    v_bits: int = 0  # value code width; 0 => bits
    symmetric: int = 0  # 1: symmetric per-token int8 keys and values (zero point 0, no residual)
    k_outliers: int = 0  # symmetric scheme: key entries per token isolated in a sparse side list
    notes: str = field(default="", compare=False)

    @property
    def vbits(self) -> int:
        return self.v_bits or self.bits

    @property
    def n_q(self) -> int:
        return self.n_kv * self.gqa

    @property
    def r_eff(self) -> int:
        if self.symmetric:
            return 1
        return self.residual if self.residual > 0 else self.k_group

    @property
    def max_seq(self) -> int:
        return self.seq + self.steps

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d_head)


WORKLOADS: dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny-int8", 1, 1, 4, 128, 1, 256, 1, 8, 32, 128, 0, 2, 20, 20260,
                 notes="oracle-sized: one layer, one kv head, GQA 4, int8, K groups of 32, V groups of 128"),
        Workload("llama8b-int8", 32, 8, 4, 128, 1, 4096, 64, 8, 128, 128, 0, 4, 20, 20261,
                 notes="Llama-style 8B cache, int8, batch 1, 4096-token prompt, 64 decode steps"),
        Workload("kivi-int4", 32, 8, 4, 128, 16, 8192, 32, 4, 128, 64, 128, 4, 20, 20262,
                 notes="KIVI-style int4, batch 16, 8192-token prompt, 128-token residual"),
        Workload("kivi-int2", 32, 8, 4, 128, 64, 4096, 32, 2, 32, 32, 128, 6, 50, 20263,
                 notes="KIVI-style int2, batch 64, 4096-token prompt, K groups of 32, 6 outlier channels x50"),
        Workload("long-int4-16k", 32, 8, 8, 128, 8, 16384, 32, 4, 128, 128, 128, 4, 20, 20264,
                 notes="long-context int4 sweep, GQA 8, 16k x batch 8"),
        Workload("long-int4-32k", 32, 8, 8, 128, 4, 32768, 32, 4, 128, 128, 128, 4, 20, 20264,
                 notes="long-context int4 sweep, GQA 8, 32k x batch 4"),
        Workload("long-int4-64k", 32, 8, 8, 128, 2, 65536, 32, 4, 128, 128, 128, 4, 20, 20264,
                 notes="long-context int4 sweep, GQA 8, 65536 x batch 2"),
        Workload("kivi-k8v4", 32, 8, 4, 128, 16, 8192, 32, 8, 128, 64, 128, 4, 20, 20265, v_bits=4,
                 notes="mixed widths: int8 keys, int4 values; otherwise the KIVI-style int4 shape"),
        Workload("llama8b-sym8", 32, 8, 4, 128, 1, 4096, 64, 8, 128, 128, 0, 4, 20, 20266, symmetric=1,
                 notes="symmetric per-token int8 keys and values; otherwise the Llama-style 8B shape"),
        Workload("sym8-b16", 32, 8, 4, 128, 16, 8192, 32, 8, 128, 128, 0, 4, 20, 20267, symmetric=1,
                 notes="symmetric per-token int8 keys and values, batch 16, 8192-token prompt"),
        Workload("sym8o4-b16", 32, 8, 4, 128, 16, 8192, 32, 8, 128, 128, 0, 4, 20, 20268, symmetric=1, k_outliers=4,
                 notes="sym8-b16 with 4 key entries per token isolated in a sparse side list"),
        Workload("kivi-int4o4", 32, 8, 4, 128, 16, 8192, 32, 4, 128, 64, 128, 4, 20, 20269, k_outliers=4,
                 notes="kivi-int4 with 4 entries of every quantized key row isolated before the per-channel groups"),
    ]
}


def k_slice(w: Workload, layer: int, b: int, h: int, tokens) -> np.ndarray:
    """Keys of one (batch row, kv head) over ``tokens``: [len(tokens)][d] binary16."""
    full = gen_k(w.seed, layer, [b], tokens, w.n_kv, w.d_head, w.n_out, w.gain, w.shift, heads=[h])
    return np.ascontiguousarray(full[0, :, 0, :])


def v_slice(w: Workload, layer: int, b: int, h: int, tokens) -> np.ndarray:
    full = gen_v(w.seed, layer, [b], tokens, w.n_kv, w.d_head, heads=[h])
    return np.ascontiguousarray(full[0, :, 0, :])


def q_rows(w: Workload, layer: int, b: int, h: int, step_token: int) -> np.ndarray:
    """The r query heads of kv head h for one batch row: [r][d] binary16."""
    q = gen_q(w.seed, layer, [b], step_token, w.n_q, w.d_head)[0]
    return np.ascontiguousarray(q[h * w.gqa:(h + 1) * w.gqa])
