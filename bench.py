#!/usr/bin/env python
"""Benchmark of the quantized-KV decode hot path on GB300.

One step = one decode step of the whole model's KV path: for every layer, append
the new token (values quantized per token, key into the binary16 residual) and run
the fused-dequant split-K decode attention over all cached tokens. Inputs (the
packed cache, the new K/V rows and the queries of every step) are resident in HBM
before the timed region; the cache of all layers (>= 280 MB) is larger than L2, so
no flush is needed between steps.

Prints ONE JSON line (rank 0). ``--impl reference`` times the CPU oracle instead,
on a bounded sample of the same workload.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import shutil
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "quantized-KV decode attention HBM GB/s (% of GB300 peak), tokens/s"
DEFAULT_WORKLOAD = "kivi-int2"  # the largest single-GPU workload: int2, batch 64 x 4096 tokens


# ----------------------------------------------------------------------------- byte accounting
def key_meta_bytes(w, n_keys: int) -> int:
    """Key metadata of n_keys quantized tokens of one slice: (scale, zero point) per channel
    and group of k_group tokens, or in the symmetric scheme one binary16 scale per token;
    plus 4 bytes (channel, binary16 value) per isolated key entry."""
    iso = n_keys * 4 * w.k_outliers  # isolated entries of the quantized key rows
    return n_keys * 2 + iso if w.symmetric else (n_keys // w.k_group) * w.d_head * 4 + iso


def attn_bytes_per_layer(w, T: int) -> int:
    """Algorithmic bytes one decode-attention launch (one layer) moves at T cached tokens:
    packed key codes + key metadata of the quantized tokens, binary16 residual keys,
    packed value codes + value metadata of all tokens, queries read, outputs written."""
    d, b, bv = w.d_head, w.bits, w.vbits
    R = w.r_eff
    Tq = (T // R) * R
    per_slice = (Tq * (d * b // 8) + key_meta_bytes(w, Tq) + (T - Tq) * 2 * d + T * (d * bv // 8)
                 + T * (d // w.v_group) * 4)
    return w.batch * w.n_kv * per_slice + w.batch * w.n_q * d * 2 + w.batch * w.n_q * d * 4


def append_bytes_per_layer(w, s_cur: int, n_new: int = 1) -> int:
    """Bytes of one append: new K/V rows read, value codes + metadata written, key rows
    written to the residual, and (when a window fills) the flushed groups re-read and packed."""
    d, b, bv = w.d_head, w.bits, w.vbits
    R = w.r_eff
    T = s_cur + n_new
    A0, A1 = (s_cur // R) * R, (T // R) * R
    per = n_new * (2 * d * 2 + d * bv // 8 + (d // w.v_group) * 4)
    per += max(0, T - max(A1, s_cur)) * 2 * d  # residual writes
    if A1 > A0:
        per += (s_cur - A0) * 2 * d + (A1 - A0) * (d * b // 8) + key_meta_bytes(w, A1 - A0)
    return w.batch * w.n_kv * per


def prefill_bytes_per_layer(w, S: int) -> int:
    """Algorithmic bytes of quantizing an S-token prompt of one layer: binary16 keys and
    values read; key codes + group metadata, residual keys, value codes + metadata written."""
    d, b, bv = w.d_head, w.bits, w.vbits
    Tq = (S // w.r_eff) * w.r_eff
    per = S * 2 * d * 2 + Tq * (d * b // 8) + key_meta_bytes(w, Tq) + (S - Tq) * 2 * d
    per += S * (d * bv // 8) + S * (d // w.v_group) * 4
    return w.batch * w.n_kv * per


def step_launches(w, s_cur: int, fused: bool = True) -> int:
    """Kernels one decode step launches: per layer one fused append+attention launch, or
    (separate calls, or a step that fills a residual window) append (+ key groups) and attention."""
    if w.symmetric:  # no residual window: the fused step is always one launch; separately key + value + attention
        return w.n_layers if fused else 3 * w.n_layers
    R = w.r_eff
    flush = ((s_cur + 1) // R) > (s_cur // R)
    if fused and not flush:
        return w.n_layers
    return w.n_layers * (2 + (1 if flush else 0))


# ----------------------------------------------------------------------------- helpers
def max_over_ranks(value: float, dist=None, device="cpu") -> float:
    """The largest value over all ranks (the slowest rank's time); identity on one rank."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, seconds: float) -> float:
    """Replicas: every rank processes the same work, so the job rate is world x units / max time."""
    return units_per_rank * world / seconds


# every source the decode-attention kernel is compiled from (its own header, the merge, and
# the shared layout, parameter and quantizer headers its fused append step uses)
DECODE_SOURCES = tuple(
    "bit_kv_cache_09_gb300/csrc/" + f
    for f in ("kvq_decode_mma.cuh", "kvq_merge.cuh", "kvq_quantizer.cuh", "kvq_common.cuh", "kvq_kernels.h",
              "kvq_decode_mma_b2.cu", "kvq_decode_mma_b4.cu", "kvq_decode_mma_b8.cu"))


def decode_source_hash() -> str:
    import hashlib

    h = hashlib.sha256()
    for f in DECODE_SOURCES:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def measured_traffic(workload: str):
    """DRAM bytes per decode-attention launch from the committed ncu capture, or None
    when there is none for this workload or the kernel source changed since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            e = json.load(f).get(workload)
    except Exception:
        return None
    if not e or e.get("kernel_src_sha") != decode_source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi samples during the timed region (SM clock, max clock, throttle reasons)."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen([exe, f"--id={self.index}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if not self.path or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": reasons, "samples": len(rows)}


# ----------------------------------------------------------------------------- CPU oracle timing
def _slice_bytes(w, T: int) -> int:
    d, bits, vbits = w.d_head, w.bits, w.vbits
    R = w.r_eff
    Tq = (T // R) * R
    return (Tq * (d * bits // 8) + key_meta_bytes(w, Tq) + (T - Tq) * 2 * d + T * (d * vbits // 8)
            + T * (d // w.v_group) * 4 + w.gqa * d * 6)


def oracle_prepare(w, layer: int, T: int, n_slices: int, budget_s: float = float("inf")):
    """Packed oracle states (the cache after T tokens) and queries of the first n_slices
    (b, h) slices of one layer. The oracle's quantization of each slice's T tokens (its
    prefill) is timed; the host generator that makes the binary16 inputs is not.
    Returns (prepared, prefill seconds, prefill algorithmic bytes)."""
    import oracle

    out, t_pre, b_pre = [], 0.0, 0
    for idx in range(min(n_slices, w.batch * w.n_kv)):
        b, h = divmod(idx, w.n_kv)
        k = synth.k_slice(w, layer, b, h, range(T))
        v = synth.v_slice(w, layer, b, h, range(T))
        t0 = time.perf_counter()
        if w.symmetric:
            st = oracle.cache_state_sym(k, v, d=w.d_head, k_outliers=w.k_outliers)
        else:
            st = oracle.cache_state(k, v, d=w.d_head, bits=w.bits, G=w.k_group, Gv=w.v_group, R=w.residual,
                                    v_bits=w.vbits, k_outliers=w.k_outliers)
        t_pre += time.perf_counter() - t0
        b_pre += prefill_bytes_per_layer(w, T) // (w.batch * w.n_kv)
        out.append((st, synth.q_rows(w, layer, b, h, T - 1)))
        if t_pre >= budget_s:
            break
    return out, t_pre, b_pre


def oracle_decode(w, prepared, budget_s: float = float("inf")):
    """Time the oracle's decode attention (dequantize the packed slice, then exact softmax
    attention in float64; single-threaded) over prepared slices. Returns (s, bytes, slices)."""
    import oracle

    total_t, total_b, n = 0.0, 0, 0
    for st, q in prepared:
        t0 = time.perf_counter()
        if w.symmetric:
            kh, vh = oracle.dequantize_state_sym(st, d=w.d_head)
        else:
            kh, vh = oracle.dequantize_state(st, d=w.d_head, bits=w.bits, G=w.k_group, Gv=w.v_group, R=w.residual,
                                             v_bits=w.vbits)
        oracle.attention(q, kh, vh, w.softmax_scale)
        total_t += time.perf_counter() - t0
        total_b += _slice_bytes(w, st.T)
        n += 1
        if total_t >= budget_s:
            break
    return total_t, total_b, n


def cpu_desc():
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for line in out.splitlines():
            if line.startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return "unknown"


def host_cores() -> int:
    """Cores of this host (nproc)."""
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 0


def workload_config(w, L: int, S: int) -> dict:
    """The workload keys of `config`, shared by both arms' lines."""
    return {"workload": w.name, "layers": L, "batch": w.batch, "n_kv_heads": w.n_kv, "gqa": w.gqa,
            "d_head": w.d_head, "prompt_tokens": S, "bits": w.bits, "v_bits": w.vbits, "symmetric": w.symmetric,
            "k_outliers": w.k_outliers, "k_group": w.k_group, "v_group": w.v_group, "residual": w.residual}


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    T = w.seq + 1
    # one step = the oracle's decode attention over a fixed sample of (b, h) slices of layer 0
    prepared, _, _ = oracle_prepare(w, 0, T, int(os.environ.get("KVQ_REF_SLICES", "4")))
    for _ in range(args.warmup):
        oracle_decode(w, prepared[:1])
    times, nbytes, slices = [], 0, 0
    for _ in range(args.steps):
        t, b, n = oracle_decode(w, prepared)
        times.append(t)
        nbytes += b
        slices = n
    total = sum(times)
    gbs = nbytes / total / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": "GB/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * total / args.steps, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {**workload_config(w, w.n_layers, w.seq), "layers_timed": 1, "T": T,
                       "sample": f"{slices} (batch row, kv head) slices of layer 0 per step"},
            "cpu_baseline": {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "host_cores": host_cores(),
                             "kind": "oracle",
                             "sample": f"oracle decode attention (dequantize packed slice + float64 softmax attention) over {slices} (b,h) slices of layer 0 at T={T}, single-threaded; CPU {cpu_desc()}"},
            "e2e": {"value": round(gbs, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------------------- GPU arm
def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="kvq", choices=["kvq", "reference"])
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--decode", default="auto", choices=["auto", "simt", "mma"])
    ap.add_argument("--no-graph", action="store_true", help="launch eagerly instead of replaying one CUDA graph per step")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle time for cpu_baseline")
    ap.add_argument("--layers", type=int, default=0, help="override the layer count (profiling only)")
    args = ap.parse_args()
    w = synth.WORKLOADS[args.workload]
    if args.layers:
        w = synth.Workload(**{**w.__dict__, "n_layers": args.layers})
    if args.impl == "reference":
        return run_reference(args, w)

    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")

    from bit_kv_cache_09_gb300 import build as kvq_build
    from bit_kv_cache_09_gb300 import kvq
    from bit_kv_cache_09_gb300.cache import QuantizedKVCache
    from synth.device import DeviceGenerator

    if rank == 0:
        kvq_build.build()
    if dist:
        dist.barrier()
    impl = {"auto": kvq.DECODE_AUTO, "simt": kvq.DECODE_SIMT, "mma": kvq.DECODE_MMA}[args.decode]
    W, K = args.warmup, args.steps
    WE, KE = (0, 0) if args.no_e2e else (2, max(3, K // 2))
    n_steps = W + K + WE + KE
    w_run = synth.Workload(**{**w.__dict__, "steps": max(w.steps, n_steps)})
    dev = torch.device("cuda", local)
    cache = QuantizedKVCache.for_workload(w_run, device=dev)
    gen = DeviceGenerator(w_run, device=dev)
    stream = torch.cuda.current_stream()
    S, L = w.seq, w.n_layers

    # prefill every layer, in chunks to bound the fp16 staging memory; the quantize-append
    # calls (not the input generator) are timed with CUDA events for the prefill line
    chunk = max(128, min(S, (1 << 28) // (w.batch * w.n_kv * w.d_head * 2) // 128 * 128))
    # one untimed append of the first chunk's shape into a one-layer scratch cache, so that
    # the timed prefill does not include loading the append kernels' code on first use
    warm = QuantizedKVCache.for_workload(synth.Workload(**{**w_run.__dict__, "seq": chunk, "steps": 0}), n_layers=1,
                                         device=dev)
    k, v = gen.kv(0, 0, min(chunk, S))
    warm.append(0, 0, k, v)
    torch.cuda.synchronize()
    del warm, k, v
    # a layer's chunks are generated first, then appended back to back between two events,
    # so that the host's per-call latency overlaps the previous call's kernels
    pre_ms = 0.0
    for layer in range(L):
        chunks = [(t, *gen.kv(layer, t, min(chunk, S - t))) for t in range(0, S, chunk)]
        p0, p1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        p0.record()
        for t, k, v in chunks:
            cache.append(layer, t, k, v)
        p1.record()
        p1.synchronize()
        pre_ms += p0.elapsed_time(p1)
        del chunks
    pre_bytes = L * prefill_bytes_per_layer(w, S)
    # inputs of every decode step, resident on the device
    kin = torch.empty((n_steps, L, w.batch, 1, w.n_kv, w.d_head), dtype=torch.float16, device=dev)
    vin = torch.empty_like(kin)
    qin = torch.empty((n_steps, L, w.batch, w.n_q, w.d_head), dtype=torch.float16, device=dev)
    for s in range(n_steps):
        for layer in range(L):
            gen.kv(layer, S + s, 1, out_k=kin[s, layer], out_v=vin[s, layer])
            gen.q(layer, S + s, out=qin[s, layer])
    out = torch.empty((L, w.batch, w.n_q, w.d_head), dtype=torch.float32, device=dev)
    torch.cuda.synchronize()
    scale = w.softmax_scale

    def step(s):
        T = S + s
        for layer in range(L):
            if impl == kvq.DECODE_SIMT:
                cache.append(layer, T, kin[s, layer], vin[s, layer])
                cache.attention(layer, T + 1, qin[s, layer], scale, out=out[layer], impl=impl)
            else:  # append fused into the attention launch
                cache.decode_step(layer, T, kin[s, layer], vin[s, layer], qin[s, layer], scale, out=out[layer])

    use_graph = not args.no_graph
    graphs = {}
    if use_graph:
        # one graph per step (s_cur differs per step); capture records launches only,
        # the cache state advances on replay
        for s in range(W + K):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(s)
            graphs[s] = g
        torch.cuda.synchronize()

    def run(s):
        if use_graph:
            graphs[s].replay()
        else:
            step(s)

    for s in range(W):
        run(s)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    launches = 0
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        e0.record()
        for s in range(W, W + K):
            run(s)
            launches += step_launches(w, S + s, fused=impl != kvq.DECODE_SIMT)
        e1.record()
        torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), dist, dev)
    clocks = clk.summary()
    nbytes = sum(L * (attn_bytes_per_layer(w, S + s + 1) + append_bytes_per_layer(w, S + s)) for s in range(W, W + K))
    ms_step = ms / K
    gbs = whole_job_rate(nbytes, world, ms / 1e3) / 1e9
    tok_s = whole_job_rate(w.batch * K, world, ms / 1e3)
    peak, peak_kind = measured_peaks()

    # dominant kernel alone: decode attention over all layers back to back (one graph), same T
    T_k = S + W + K
    reps = 5
    ga = torch.cuda.CUDAGraph()
    with torch.cuda.graph(ga):
        for layer in range(L):
            cache.attention(layer, T_k, qin[W + K - 1, layer], scale, out=out[layer], impl=impl)
    ga.replay()
    torch.cuda.synchronize()
    a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a0.record()
    for _ in range(reps):
        ga.replay()
    a1.record()
    torch.cuda.synchronize()
    attn_us = a0.elapsed_time(a1) * 1e3 / (reps * L)
    attn_b = attn_bytes_per_layer(w, T_k)
    achieved = attn_b / (attn_us * 1e-6) / 1e9
    traffic = measured_traffic(w.name)

    # end to end through the public API: pinned host inputs in, outputs back, every step
    e2e = None
    if KE:
        kh = kin[W + K:].cpu().pin_memory()
        vh = vin[W + K:].cpu().pin_memory()
        qh = qin[W + K:].cpu().pin_memory()
        oh = torch.empty((KE + WE, L, w.batch, w.n_q, w.d_head), dtype=torch.float32).pin_memory()
        kd = torch.empty_like(kin[0])
        vd = torch.empty_like(vin[0])
        qd = torch.empty_like(qin[0])

        def e2e_step(i):
            s = W + K + i
            T = S + s
            kd.copy_(kh[i], non_blocking=True)
            vd.copy_(vh[i], non_blocking=True)
            qd.copy_(qh[i], non_blocking=True)
            for layer in range(L):
                if impl == kvq.DECODE_SIMT:
                    cache.append(layer, T, kd[layer], vd[layer])
                    cache.attention(layer, T + 1, qd[layer], scale, out=out[layer], impl=impl)
                else:
                    cache.decode_step(layer, T, kd[layer], vd[layer], qd[layer], scale, out=out[layer])
            oh[i].copy_(out, non_blocking=True)

        # one graph per step: host->device copies of the step's inputs (pinned), the
        # decode step of every layer, and the device->host copy of the outputs
        e2e_graphs = {}
        if use_graph:
            for i in range(WE + KE):
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g):
                    e2e_step(i)
                e2e_graphs[i] = g
            torch.cuda.synchronize()

        def e2e_run(i):
            if use_graph:
                e2e_graphs[i].replay()
            else:
                e2e_step(i)

        for i in range(WE):
            e2e_run(i)
        torch.cuda.synchronize()
        b0, b1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t_host = time.perf_counter()
        b0.record()
        for i in range(WE, WE + KE):
            e2e_run(i)
        b1.record()
        torch.cuda.synchronize()
        t_host = time.perf_counter() - t_host
        e_ms = max(b0.elapsed_time(b1), t_host * 1e3)
        e_bytes = sum(L * (attn_bytes_per_layer(w, S + W + K + i + 1) + append_bytes_per_layer(w, S + W + K + i))
                      for i in range(WE, WE + KE))
        h2d = (kd.numel() + vd.numel() + qd.numel()) * 2
        d2h = out.numel() * 4
        e2e = {"value": round(e_bytes * world / (e_ms / 1e3) / 1e9, 2), "unit": "GB/s",
               "tokens_per_s": round(w.batch * KE * world / (e_ms / 1e3), 1),
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": KE, "cuda_graph": use_graph,
               "device_ms": round(b0.elapsed_time(b1), 3), "host_ms": round(t_host * 1e3, 3)}

    cache.check_errors()  # no bounded wait of any timed launch ran out
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        # the oracle as it stands, single-threaded: prefill quantization of layer 0's
        # slices (the prompt), then their decode attention, each within half the budget
        prepared, tp, bp = oracle_prepare(w, 0, S + 1, 8, args.cpu_budget / 2)
        t, b, n = oracle_decode(w, prepared, args.cpu_budget / 2)
        slices = w.batch * w.n_kv
        cpu = {"value": round(b / t / 1e9, 5), "unit": "GB/s", "cores": 1, "host_cores": host_cores(),
               "kind": "oracle",
               "sample": f"oracle decode attention of layer 0 (dequantize packed slice + float64 softmax attention), {n} of {slices} (b,h) slices at T={S + 1}, single-threaded; CPU {cpu_desc()}",
               "us_per_slice": round(t / n * 1e6, 1),
               "step_s_extrapolated": round(t / n * slices * L, 3),
               "prefill": {"value": round(bp / tp / 1e9, 5), "unit": "GB/s",
                           "sample": f"oracle quantization of the {S + 1}-token prompt of layer 0, {len(prepared)} (b,h) slices (binary16 keys and values read, codes, metadata and residual written), single-threaded"}}

    if rank == 0:
        line = {"metric": METRIC, "value": round(gbs, 2), "unit": "GB/s", "n_gpus": world, "steps": K, "warmup": W,
                "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": ((f"int8 symmetric per-token codes + {w.k_outliers} binary16 key entries per token"
                           if w.k_outliers else "int8 symmetric per-token codes") if w.symmetric else
                          f"int{w.bits} codes" if w.vbits == w.bits else f"int{w.bits} key / int{w.vbits} value codes")
                + ", f32 math", "data": "synthetic",
                "tokens_per_s": round(tok_s, 1), "pct_of_peak": round(100 * gbs / world / peak, 2),
                "config": {**workload_config(w, L, S), "decode": args.decode,
                           "cuda_graph": use_graph, "parallelism": f"replicas x{world}",
                           "l2": "per-step working set (all layers' packed cache) exceeds the 129 MB L2; no flush"},
                "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                             "frac": round(achieved / peak, 4), "traffic": traffic,
                             "kernel": "decode attention", "us_per_launch": round(attn_us, 3),
                             "bytes_per_launch": attn_b, "peak_kind": f"{peak_kind} hbm_gbs"},
                "prefill": {"what": f"quantize-append of the {S}-token prompt, all layers, chunks of {chunk} tokens "
                                    "(key-group and value-token kernels), CUDA events around each layer's calls",
                            "gbs": round(pre_bytes / (pre_ms / 1e3) / 1e9, 1), "frac": round(pre_bytes / (pre_ms / 1e3) / 1e9 / peak, 4),
                            "ms": round(pre_ms, 3), "bytes": pre_bytes},
                "gpu_launches": launches, "clocks": clocks, "e2e": e2e, "cpu_baseline": cpu}
        print(json.dumps(line), flush=True)
    if dist:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
