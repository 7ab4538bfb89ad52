// kvq_api.cu — the C ABI of libkvq (declared in include/kvq.h): argument checks,
// geometry, split-K planning and kernel dispatch. Host code only; every check runs
// before any launch, and a failed check launches nothing.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "kvq_common.cuh"
#include "kvq_kernels.h"

using kvq::Geometry;

namespace {

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

kvq_status check_buffers(const kvq_buffers* b) {
  if (!b) return KVQ_ERR_INVALID_ARG;
  const void* ps[5] = {b->k_codes, b->k_meta, b->k_resid, b->v_codes, b->v_meta};
  for (const void* p : ps)
    if (!aligned16(p)) return KVQ_ERR_INVALID_ARG;
  return KVQ_OK;
}

// Layer-0-relative pointers of one layer.
struct LayerPtrs {
  uint8_t* k_codes;
  __half2* k_meta;
  __half* k_resid;
  uint8_t* v_codes;
  __half2* v_meta;
};

LayerPtrs layer_ptrs(const Geometry& g, const kvq_buffers* b, int layer) {
  const int64_t s0 = (int64_t)layer * g.B * g.H;  // first slice of the layer
  LayerPtrs p;
  p.k_codes = static_cast<uint8_t*>(b->k_codes) + s0 * g.k_codes_slice;
  p.k_meta = reinterpret_cast<__half2*>(static_cast<uint8_t*>(b->k_meta) + s0 * g.k_meta_slice);
  p.k_resid = reinterpret_cast<__half*>(static_cast<uint8_t*>(b->k_resid) + s0 * g.k_resid_slice);
  p.v_codes = static_cast<uint8_t*>(b->v_codes) + s0 * g.v_codes_slice;
  p.v_meta = reinterpret_cast<__half2*>(static_cast<uint8_t*>(b->v_meta) + s0 * g.v_meta_slice);
  return p;
}

// SM count of the current device (cached per device; 0 if the query fails)
int device_sm_count() {
  static std::atomic<int> cache[16];
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 16 && (n = cache[dev].load(std::memory_order_relaxed)) > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 16) cache[dev].store(n, std::memory_order_relaxed);
  return n;
}

// Resident CTAs per SM of the decode kernel that `impl` selects (cached per device).
// Index of the (key, value) code widths: 8/8, 4/4, 2/2, 8/4.
int width_index(const Geometry& g) {
  if (g.sym) return g.kout > 0 ? 5 : 4;  // symmetric per-token int8 (with isolated key entries)
  const int w = g.vbits != g.bits ? 3 : (g.bits == 8 ? 0 : (g.bits == 4 ? 1 : 2));
  return g.kout > 0 ? 6 + w : w;  // per-channel keys, with isolated key entries: 6..9
}

// Kernel family of the occupancy queries: 0 asymmetric, 1 symmetric, 2 symmetric with
// isolated key entries, 3 asymmetric with isolated key entries.
int scheme(const Geometry& g) { return g.sym ? (g.kout > 0 ? 2 : 1) : (g.kout > 0 ? 3 : 0); }

int decode_occupancy(const Geometry& g, kvq_decode_impl impl) {
  static std::atomic<int> cache[16][2][10][2][3];  // device, impl, code scheme/widths, r class, value groups
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) dev = 0;
  const int ii = impl == KVQ_DECODE_SIMT ? 0 : 1;
  const int bi = width_index(g);
  const int ri = g.r <= 4 ? 0 : 1;
  const int vi = g.n_vg == 1 ? 0 : (g.n_vg == 2 ? 1 : 2);
  std::atomic<int>& slot = cache[dev][ii][bi][ri][vi];
  int n = slot.load(std::memory_order_relaxed);
  if (n <= 0) {
    n = ii == 0 ? kvq::occupancy_decode_simt(g.bits)
                : kvq::occupancy_decode_mma(g.bits, g.vbits, g.r, g.n_vg, scheme(g));
    if (n > 0) slot.store(n, std::memory_order_relaxed);
  }
  return n > 0 ? n : 1;
}

// Clusters of `cs` CTAs (a power of two, 2..16) of `nw` warps of the tensor-core
// kernel that can be resident at once on this device (<= 0: such a cluster cannot
// launch); cached per device and kernel shape.
int resident_clusters(const Geometry& g, int cs, int nw) {
  static std::atomic<int> cache[16][10][2][3][5][3];  // device, code scheme/widths, r class, value groups, log2 size, warps
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 16) dev = 0;
  const int bi = width_index(g);
  const int ri = g.r <= 4 ? 0 : 1;
  const int vi = g.n_vg == 1 ? 0 : (g.n_vg == 2 ? 1 : 2);
  int lg = 0;
  while ((1 << lg) < cs) ++lg;
  std::atomic<int>& slot = cache[dev][bi][ri][vi][lg][nw == 8 ? 2 : (nw == 5 ? 1 : 0)];
  int n = slot.load(std::memory_order_relaxed);
  if (n == 0) {
    n = kvq::max_clusters_decode_mma(g.bits, g.vbits, g.r, g.n_vg, cs, nw, scheme(g));
    if (n <= 0) n = -1;
    slot.store(n, std::memory_order_relaxed);
  }
  return n;
}

// Largest power-of-two cluster size <= 16 whose clusters of nw-warp CTAs can all be
// resident for `units` (batch row, kv head) pairs (1: none).
int decode_cluster_size(const Geometry& g, int64_t units, int nw) {
  for (int lg = 4; lg >= 1; --lg)
    if (resident_clusters(g, 1 << lg, nw) >= units) return 1 << lg;
  return 1;
}

// Split-K plan.
// Large grids (many (batch row, kv head) pairs): the number of splits per pair minimises
// a cost model (rounds of resident CTAs x per-CTA time); 2, 4 or 8 splits of a pair run
// as one cluster and merge through distributed shared memory, other counts merge
// through the workspace (last CTA, atomic ticket).
// Small grids (at most 1/32 of the slots per pair): latency-bound, so each pair gets a
// cluster of up to 16 CTAs, small enough that every warp's stages are all in flight at
// once, merged through distributed shared memory without touching the workspace; CTAs
// of 5 or 8 warps are used when that shortens the longest warp's run of iterations.
struct Plan {
  int64_t n_split, chunk;
  int cluster, n_parts;
  int warps = 4;
  // mixed plan: the first pairs_hi pairs take n_split splits of `chunk` tokens, the others
  // n_split - 1 splits of chunk_lo tokens; every pair merges through the workspace
  int mixed = 0;
  int pairs_hi = 0;
  int64_t chunk_lo = 0;
};

Plan plan_splits(const Geometry& g, int64_t T, kvq_decode_impl impl) {
  int sms = device_sm_count();
  if (sms <= 0) sms = 152;
  const int64_t slots = (int64_t)sms * decode_occupancy(g, impl);
  const int64_t align = impl == KVQ_DECODE_SIMT ? 128 : 32;
  const int64_t units = (int64_t)g.B * g.H;
  Plan pl;
  if (impl != KVQ_DECODE_SIMT && units * 32 <= slots) {
    int64_t best_run = -1;
    for (int nw : {4, 5, 8}) {
      const int cs = decode_cluster_size(g, units, nw);
      if (nw != 4 && cs < 2) continue;
      int64_t c = (T + cs - 1) / cs;
      c = (c + align - 1) / align * align;
      const int64_t run = (c / 32 + nw - 1) / nw;  // iterations of the busiest warp
      if (best_run < 0 || run < best_run) {
        best_run = run;
        pl.n_split = cs;  // trailing splits may be empty; they merge with weight 0
        pl.chunk = c;
        pl.cluster = cs;
        pl.n_parts = 1;
        pl.warps = nw;
      }
    }
    return pl;
  }
  int64_t max_k = kvq::max_splits(g, T);
  const int64_t by_len = (T + align - 1) / align;
  if (max_k > by_len) max_k = by_len;
  if (max_k < 1) max_k = 1;
  // Cost model: the CTAs of a split run in rounds of `slots` co-resident CTAs; a round
  // lasts as long as one CTA: a fixed cost (prologue, pipeline fill, merge; about four
  // loop iterations of a warp, measured) plus its loop iterations (each of the 4 warps
  // takes 32 tokens per iteration). Ties go to fewer splits.
  const int64_t per_it = 128;
  const int64_t fixed_it = 4;
  int64_t best_cost = -1, best_chunk = align;
  for (int64_t k = 1; k <= max_k; ++k) {
    int64_t c = (T + k - 1) / k;
    c = (c + align - 1) / align * align;
    const int64_t n = (T + c - 1) / c;
    const int64_t rounds = (units * n + slots - 1) / slots;
    const int64_t cost = rounds * (fixed_it + (c + per_it - 1) / per_it);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best_chunk = c;
    }
  }
  const int64_t c = best_chunk;
  pl.n_split = (T + c - 1) / c;
  pl.chunk = c;
  pl.cluster = 1;
  pl.n_parts = (int)pl.n_split;
  if (impl != KVQ_DECODE_SIMT && (pl.n_split == 2 || pl.n_split == 4 || pl.n_split == 8) &&
      resident_clusters(g, (int)pl.n_split, 4) > 0) {
    pl.cluster = (int)pl.n_split;
    pl.n_parts = 1;
  }
  // Balanced alternative (tensor-core kernel): fill the resident slots exactly, k splits for
  // most pairs and k + 1 for the rest. The loop is bound by instruction issue per SM, so a
  // launch lasts as long as its busiest SM's share of work, and with equal splits that do
  // not fill the slots some SMs hold one CTA more than others. Busiest SM, in warp
  // iterations, with CTAs spread over the SMs in launch order: the uniform plan's
  // ceil(CTAs / SMs) CTAs; the mixed plan's ceil(long CTAs / SMs) long and the rest short
  // ones. Ties keep the uniform plan, and so does a uniform plan that merges its splits in
  // clusters: measured on GB300, the balance then does not pay for the workspace merge
  // (kivi-int4 +0.5 %, kivi-k8v4 -3 %), while it does against one split per pair
  // (kivi-int2 +9 %).
  if (impl != KVQ_DECODE_SIMT && pl.cluster == 1) {
    const int64_t occ = slots / sms;
    const int64_t k = slots / units;  // splits of most pairs
    const int64_t pairs_hi = slots - units * k;
    auto warp_iters = [&](int64_t chunk) { return (chunk / 32 + 3) / 4; };
    auto chunk_of = [&](int64_t splits) { return ((T + splits - 1) / splits + align - 1) / align * align; };
    if (k >= 1 && pairs_hi > 0 && k + 1 <= max_k) {
      const int64_t c_hi = chunk_of(k + 1), c_lo = chunk_of(k);
      if ((T + c_hi - 1) / c_hi == k + 1 && (T + c_lo - 1) / c_lo == k) {
        const int64_t n_long = (units - pairs_hi) * k;
        const int64_t per_sm_long = std::min<int64_t>(occ, (n_long + sms - 1) / sms);
        const int64_t mixed_cost = per_sm_long * (fixed_it + warp_iters(c_lo)) +
                                   (occ - per_sm_long) * (fixed_it + warp_iters(c_hi));
        const int64_t n_uni = units * pl.n_split;
        const int64_t uni_cost = n_uni <= slots ? ((n_uni + sms - 1) / sms) * (fixed_it + warp_iters(pl.chunk))
                                                : ((n_uni + slots - 1) / slots) * occ * (fixed_it + warp_iters(pl.chunk));
        if (mixed_cost < uni_cost) {
          pl.mixed = 1;
          pl.n_split = k + 1;
          pl.chunk = c_hi;
          pl.chunk_lo = c_lo;
          pl.pairs_hi = (int)pairs_hi;
          pl.cluster = 1;
          pl.n_parts = (int)(k + 1);
        }
      }
    }
  }
  return pl;
}

}  // namespace

extern "C" {

const char* kvq_status_string(kvq_status s) {
  switch (s) {
    case KVQ_OK: return "ok";
    case KVQ_ERR_INVALID_ARG: return "invalid argument";
    case KVQ_ERR_UNSUPPORTED: return "unsupported configuration";
    case KVQ_ERR_CAPACITY: return "cache capacity exceeded";
    case KVQ_ERR_WORKSPACE: return "workspace missing or too small";
    case KVQ_ERR_CUDA: return "CUDA launch error";
  }
  return "unknown status";
}

const char* kvq_version(void) { return "kvq 0.1.0 sm_103a"; }

kvq_status kvq_buffer_sizes(const kvq_config* cfg, size_t bytes[KVQ_NUM_BUFFERS]) {
  if (!bytes) return KVQ_ERR_INVALID_ARG;
  Geometry g;
  kvq_status st = kvq::make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  bytes[KVQ_BUF_K_CODES] = (size_t)(g.n_slices * g.k_codes_slice);
  bytes[KVQ_BUF_K_META] = (size_t)(g.n_slices * g.k_meta_slice);
  bytes[KVQ_BUF_K_RESID] = (size_t)(g.n_slices * g.k_resid_slice);
  bytes[KVQ_BUF_V_CODES] = (size_t)(g.n_slices * g.v_codes_slice);
  bytes[KVQ_BUF_V_META] = (size_t)(g.n_slices * g.v_meta_slice);
  return KVQ_OK;
}

kvq_status kvq_quantize_append(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                               int64_t n_new, const void* k_f16, const void* v_f16, void* stream) {
  Geometry g;
  kvq_status st = kvq::make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if ((st = check_buffers(bufs)) != KVQ_OK) return st;
  if (layer < 0 || layer >= g.L || s_cur < 0 || n_new < 1) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_f16) || !aligned16(v_f16)) return KVQ_ERR_INVALID_ARG;
  if (s_cur + n_new > g.S_max) return KVQ_ERR_CAPACITY;
  const int64_t T = s_cur + n_new;
  const int64_t A0 = (s_cur / g.R_eff) * g.R_eff;
  const int64_t A1 = (T / g.R_eff) * g.R_eff;
  const LayerPtrs lp = layer_ptrs(g, bufs, layer);
  kvq::AppendParams p;
  p.k_codes = lp.k_codes;
  p.k_meta = lp.k_meta;
  p.k_resid = lp.k_resid;
  p.v_codes = lp.v_codes;
  p.v_meta = lp.v_meta;
  p.k_in = static_cast<const __half*>(k_f16);
  p.v_in = static_cast<const __half*>(v_f16);
  p.s_cur = s_cur;
  p.n_new = n_new;
  p.A1 = A1;
  p.group0 = A0 / g.G;
  p.n_groups = (int)((A1 - A0) / g.G);
  p.B = g.B;
  p.H = g.H;
  p.G = g.G;
  p.Gv = g.Gv;
  p.R_eff = g.R_eff;
  p.n_vg = g.n_vg;
  p.S_pad = g.S_pad;
  p.rowK = g.rowK;
  p.rowV = g.rowV;
  p.k_codes_slice = g.k_codes_slice;
  p.k_meta_slice = g.k_meta_slice;
  p.kout = g.kout;
  p.v_codes_slice = g.v_codes_slice;
  p.fd_H = kvq::make_fast_div((uint32_t)g.H);
  p.rows_32 = n_new * g.H < (int64_t(1) << 31);
  p.sym = g.sym;
  p.wide_keys = g.kout > 0;
  cudaError_t e = kvq::launch_append(p, g.bits, g.vbits, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

kvq_status kvq_dequantize(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur, float* k_out,
                          float* v_out, void* stream) {
  Geometry g;
  kvq_status st = kvq::make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if ((st = check_buffers(bufs)) != KVQ_OK) return st;
  if (layer < 0 || layer >= g.L || s_cur < 1) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_out) || !aligned16(v_out)) return KVQ_ERR_INVALID_ARG;
  if (s_cur > g.S_max) return KVQ_ERR_CAPACITY;
  const LayerPtrs lp = layer_ptrs(g, bufs, layer);
  kvq::DequantParams p;
  p.k_codes = lp.k_codes;
  p.k_meta = lp.k_meta;
  p.k_resid = lp.k_resid;
  p.v_codes = lp.v_codes;
  p.v_meta = lp.v_meta;
  p.k_out = k_out;
  p.v_out = v_out;
  p.T = s_cur;
  p.Tq = kvq::quantized_keys(g, s_cur);
  p.B = g.B;
  p.H = g.H;
  p.G = g.G;
  p.Gv = g.Gv;
  p.R_eff = g.R_eff;
  p.n_vg = g.n_vg;
  p.S_pad = g.S_pad;
  p.rowK = g.rowK;
  p.rowV = g.rowV;
  p.k_codes_slice = g.k_codes_slice;
  p.k_meta_slice = g.k_meta_slice;
  p.kout = g.kout;
  p.v_codes_slice = g.v_codes_slice;
  p.sym = g.sym;
  cudaError_t e = kvq::launch_dequant(p, g.bits, g.vbits, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

size_t kvq_decode_workspace_size(const kvq_config* cfg, int64_t s_cur) {
  Geometry g;
  if (kvq::make_geometry(cfg, &g) != KVQ_OK || s_cur < 1) return 0;
  return kvq::workspace_layout(g, s_cur).total;
}

int32_t kvq_decode_num_splits(const kvq_config* cfg, int64_t s_cur) {
  Geometry g;
  if (kvq::make_geometry(cfg, &g) != KVQ_OK || s_cur < 1) return 0;
  return (int32_t)plan_splits(g, s_cur, KVQ_DECODE_MMA).n_split;
}

}  // extern "C"

namespace kvq {

// Checks a decode-attention call over s_cur tokens and fills its launch description;
// launches nothing. When k_new/v_new are given (tensor-core kernel only) the kernel
// first appends token s_cur - 1 itself. early: the tensor-core kernel copies its first
// cache tiles before waiting on the previous kernel of the stream
// (KVQ_DECODE_EARLY_PREFETCH). wait_ns: time limit of the kernel's bounded waits.
kvq_status decode_prepare(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                          const void* q_f16, float softmax_scale, float* out, void* ws, size_t ws_bytes,
                          kvq_decode_impl impl, const void* k_new, const void* v_new, bool early, uint64_t wait_ns,
                          DecodeCall* call) {
  Geometry g;
  kvq_status st = kvq::make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if ((st = check_buffers(bufs)) != KVQ_OK) return st;
  if (layer < 0 || layer >= g.L || s_cur < 1) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(q_f16) || !aligned16(out)) return KVQ_ERR_INVALID_ARG;
  if (!(softmax_scale == softmax_scale) || softmax_scale == __builtin_inff() || softmax_scale == -__builtin_inff())
    return KVQ_ERR_INVALID_ARG;
  if (impl != KVQ_DECODE_AUTO && impl != KVQ_DECODE_SIMT && impl != KVQ_DECODE_MMA) return KVQ_ERR_INVALID_ARG;
  if (s_cur > g.S_max) return KVQ_ERR_CAPACITY;
  const kvq::WorkspaceLayout wl = kvq::workspace_layout(g, s_cur);
  if (!aligned16(ws) || ws_bytes < wl.total) return KVQ_ERR_WORKSPACE;
  const kvq_decode_impl use = impl == KVQ_DECODE_SIMT ? KVQ_DECODE_SIMT : KVQ_DECODE_MMA;
  if (use == KVQ_DECODE_SIMT && (k_new || v_new)) return KVQ_ERR_UNSUPPORTED;
  if (use == KVQ_DECODE_SIMT && g.vbits != g.bits) return KVQ_ERR_UNSUPPORTED;  // CUDA-core kernel: equal widths
  if (use == KVQ_DECODE_SIMT && (g.sym || g.kout > 0)) return KVQ_ERR_UNSUPPORTED;  // and plain asymmetric keys
  const LayerPtrs lp = layer_ptrs(g, bufs, layer);
  kvq::DecodeParams& p = call->p;
  p = kvq::DecodeParams{};
  p.k_codes = lp.k_codes;
  p.k_meta = lp.k_meta;
  p.k_resid = lp.k_resid;
  p.v_codes = lp.v_codes;
  p.v_meta = lp.v_meta;
  p.q = static_cast<const __half*>(q_f16);
  p.k_new = static_cast<const __half*>(k_new);
  p.v_new = static_cast<const __half*>(v_new);
  p.k_resid_w = lp.k_resid;
  p.v_codes_w = lp.v_codes;
  p.v_meta_w = lp.v_meta;
  p.k_codes_w = lp.k_codes;
  p.k_meta_w = lp.k_meta;
  p.out = out;
  p.err = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + wl.err_off);
  p.wait_ns = wait_ns;
  p.tickets = reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(ws) + wl.tickets_off);
  p.ws_ml = reinterpret_cast<float2*>(static_cast<uint8_t*>(ws) + wl.ml_off);
  p.ws_o = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + wl.o_off);
  p.T = s_cur;
  p.Tq = kvq::quantized_keys(g, s_cur);
  p.cap = (int)wl.cap;
  p.B = g.B;
  p.H = g.H;
  p.r = g.r;
  p.G = g.G;
  p.log2G = g.G == 32 ? 5 : (g.G == 64 ? 6 : 7);
  p.Gv = g.Gv;
  p.R_eff = g.R_eff;
  p.n_vg = g.n_vg;
  p.S_pad = g.S_pad;
  p.rowK = g.rowK;
  p.rowV = g.rowV;
  p.k_codes_slice = g.k_codes_slice;
  p.k_meta_slice = g.k_meta_slice;
  p.kout = g.kout;
  p.v_codes_slice = g.v_codes_slice;
  p.scale_log2 = softmax_scale * 1.4426950408889634f;
  const Plan pl = plan_splits(g, s_cur, use);
  p.n_split = (int)pl.n_split;
  p.chunk = pl.chunk;
  p.cluster = pl.cluster;
  p.n_parts = pl.n_parts;
  p.warps = pl.warps;
  p.mixed = pl.mixed;
  p.n_hi = (int)pl.n_split;
  p.pairs_hi = pl.pairs_hi;
  p.chunk_hi = pl.chunk;
  p.chunk_lo = pl.chunk_lo;
  p.sym = g.sym;
  p.early = (early && use == KVQ_DECODE_MMA) ? 1 : 0;
  call->simt = use == KVQ_DECODE_SIMT;
  call->bits = g.bits;
  call->vbits = g.vbits;
  call->counters_bytes = wl.ml_off;
  return KVQ_OK;
}

kvq_status decode_enqueue(const DecodeCall& call, cudaStream_t stream) {
  const cudaError_t e = call.simt ? kvq::launch_decode_simt(call.p, call.bits, stream)
                                  : kvq::launch_decode_mma(call.p, call.bits, call.vbits, stream);
  return e == cudaSuccess ? KVQ_OK : KVQ_ERR_CUDA;
}

// Reads the error word at `err` (device) once all work enqueued before on `stream` has
// finished, stores it in *out and clears it.
kvq_status read_error_word(uint32_t* err, cudaStream_t stream, uint32_t* out) {
  if (cudaMemcpyAsync(out, err, sizeof(uint32_t), cudaMemcpyDeviceToHost, stream) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaMemsetAsync(err, 0, sizeof(uint32_t), stream) != cudaSuccess) return KVQ_ERR_CUDA;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return KVQ_ERR_CUDA;
  return KVQ_OK;
}

}  // namespace kvq

namespace {

kvq_status decode_launch(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                         const void* q_f16, float softmax_scale, float* out, void* ws, size_t ws_bytes, void* stream,
                         kvq_decode_impl impl, const void* k_new, const void* v_new, bool early,
                         uint64_t wait_ns = kvq::kDefaultWaitNs) {
  kvq::DecodeCall call;
  const kvq_status st = kvq::decode_prepare(cfg, bufs, layer, s_cur, q_f16, softmax_scale, out, ws, ws_bytes, impl,
                                            k_new, v_new, early, wait_ns, &call);
  if (st != KVQ_OK) return st;
  return kvq::decode_enqueue(call, static_cast<cudaStream_t>(stream));
}

uint64_t wait_limit(uint32_t flags) { return (flags & KVQ_DECODE_ZERO_WAIT_LIMIT) ? 0ull : kvq::kDefaultWaitNs; }

constexpr uint32_t kDecodeFlags = KVQ_DECODE_EARLY_PREFETCH | KVQ_DECODE_ZERO_WAIT_LIMIT;

}  // namespace

extern "C" {

kvq_status kvq_decode_attention_impl(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                                     const void* q_f16, float softmax_scale, float* out, void* ws,
                                     size_t ws_bytes, void* stream, kvq_decode_impl impl) {
  return decode_launch(cfg, bufs, layer, s_cur, q_f16, softmax_scale, out, ws, ws_bytes, stream, impl, nullptr,
                       nullptr, false);
}

kvq_status kvq_decode_attention_ex(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                                   const void* q_f16, float softmax_scale, float* out, void* ws, size_t ws_bytes,
                                   void* stream, uint32_t flags) {
  if (flags & ~kDecodeFlags) return KVQ_ERR_INVALID_ARG;
  return decode_launch(cfg, bufs, layer, s_cur, q_f16, softmax_scale, out, ws, ws_bytes, stream, KVQ_DECODE_AUTO,
                       nullptr, nullptr, (flags & KVQ_DECODE_EARLY_PREFETCH) != 0, wait_limit(flags));
}

kvq_status kvq_decode_step_ex(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                              const void* k_f16, const void* v_f16, const void* q_f16, float softmax_scale, float* out,
                              void* ws, size_t ws_bytes, void* stream, uint32_t flags) {
  if (flags & ~kDecodeFlags) return KVQ_ERR_INVALID_ARG;
  const bool early = (flags & KVQ_DECODE_EARLY_PREFETCH) != 0;
  Geometry g;
  kvq_status st = kvq::make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if ((st = check_buffers(bufs)) != KVQ_OK) return st;
  if (layer < 0 || layer >= g.L || s_cur < 0) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(k_f16) || !aligned16(v_f16)) return KVQ_ERR_INVALID_ARG;
  if (s_cur + 1 > g.S_max) return KVQ_ERR_CAPACITY;
  const int64_t T = s_cur + 1;
  if (!g.sym && T % g.R_eff == 0) {  // the append fills a residual window: quantize it with the append kernels
    st = kvq_quantize_append(cfg, bufs, layer, s_cur, 1, k_f16, v_f16, stream);
    if (st != KVQ_OK) return st;
    // the kernel just launched writes this layer: the attention launch waits for it
    return decode_launch(cfg, bufs, layer, T, q_f16, softmax_scale, out, ws, ws_bytes, stream, KVQ_DECODE_AUTO,
                         nullptr, nullptr, false, wait_limit(flags));
  }
  return decode_launch(cfg, bufs, layer, T, q_f16, softmax_scale, out, ws, ws_bytes, stream, KVQ_DECODE_AUTO, k_f16,
                       v_f16, early, wait_limit(flags));
}

kvq_status kvq_decode_step(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                           const void* k_f16, const void* v_f16, const void* q_f16, float softmax_scale, float* out,
                           void* ws, size_t ws_bytes, void* stream) {
  return kvq_decode_step_ex(cfg, bufs, layer, s_cur, k_f16, v_f16, q_f16, softmax_scale, out, ws, ws_bytes, stream, 0u);
}

kvq_status kvq_decode_attention(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                                const void* q_f16, float softmax_scale, float* out, void* ws, size_t ws_bytes,
                                void* stream) {
  return kvq_decode_attention_impl(cfg, bufs, layer, s_cur, q_f16, softmax_scale, out, ws, ws_bytes, stream,
                                   KVQ_DECODE_AUTO);
}

}  // extern "C"

extern "C" kvq_status kvq_decode_error(void* ws, size_t ws_bytes, void* stream, uint32_t* err_out) {
  if (!err_out) return KVQ_ERR_INVALID_ARG;
  if (!aligned16(ws) || ws_bytes < 256) return KVQ_ERR_WORKSPACE;
  return kvq::read_error_word(static_cast<uint32_t*>(ws), static_cast<cudaStream_t>(stream), err_out);
}
