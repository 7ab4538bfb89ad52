// kvq_common.cuh — cache geometry shared by the host API and the kernels of libkvq.
//
// Geometry of the packed cache (see include/kvq.h for the byte layout):
//   slice (layer l, batch row b, kv head h) = (l * B + b) * H + h
//   k_codes slice: S_pad rows of rowK = d*b/8 bytes
//   k_meta  slice: S_pad/G groups x d x half2(scale, zero_point), then (kout > 0)
//                  S_pad x kout isolated entries {channel u16, value binary16}
//   k_resid slice: R_eff rows x d binary16
//   v_codes slice: S_pad/2 pair rows of 2*rowV bytes (rowV = d*b/8)
//   v_meta  slice: S_pad/2 token pairs x d/Gv x {scale 2p, scale 2p+1, zp 2p, zp 2p+1}
// Symmetric per-token scheme: k_meta slice = S_pad binary16 key scales (then, with kout
// isolated entries per token, S_pad x kout x {channel u16, value binary16}), no k_resid,
// Gv = d (v_meta zero points are 0), every key quantized on append (Tq = T).
#pragma once

#include <cstddef>
#include <cstdint>

#include "../../include/kvq.h"

namespace kvq {

constexpr int kHeadDim = 128;     // the only d_head this build implements
constexpr int kSeqAlign = 128;    // S_pad granularity (a multiple of every group and tile size)
constexpr int kMaxGqa = 8;        // query heads per kv head handled by one CTA
constexpr int kMaxResidual = 1024;

struct Geometry {
  int L, B, H, r, d, S_max, bits, vbits, G, Gv, R, R_eff;  // bits: keys, vbits: values
  int sym;             // symmetric per-token int8 scheme
  int kout;            // isolated key entries per token (both schemes)
  int64_t S_pad;
  int64_t rowK, rowV;  // bytes per token row of key / value codes
  int n_vg;            // value groups per token (d / Gv)
  int64_t k_codes_slice, k_meta_slice, k_resid_slice, v_codes_slice, v_meta_slice;  // bytes per slice
  int64_t n_slices;    // L * B * H
};

// Validates a configuration and derives its geometry. Pure host code (no CUDA calls).
inline kvq_status make_geometry(const kvq_config* c, Geometry* g) {
  if (!c || !g) return KVQ_ERR_INVALID_ARG;
  if (c->n_layers < 1 || c->batch < 1 || c->n_kv_heads < 1 || c->gqa_ratio < 1 || c->d_head < 1 ||
      c->max_seq_len < 1 || c->k_group < 1 || c->v_group < 1 || c->residual_len < 0)
    return KVQ_ERR_INVALID_ARG;
  if (c->bits != 2 && c->bits != 4 && c->bits != 8) return KVQ_ERR_UNSUPPORTED;
  const int vbits = c->v_bits == 0 ? c->bits : c->v_bits;
  if (vbits != 2 && vbits != 4 && vbits != 8) return KVQ_ERR_UNSUPPORTED;
  if (vbits != c->bits && !(c->bits == 8 && vbits == 4)) return KVQ_ERR_UNSUPPORTED;  // mixed: 8-bit keys, 4-bit values
  if (c->d_head != kHeadDim) return KVQ_ERR_UNSUPPORTED;
  if (c->k_group != 32 && c->k_group != 64 && c->k_group != 128) return KVQ_ERR_UNSUPPORTED;
  if (c->v_group != 32 && c->v_group != 64 && c->v_group != 128) return KVQ_ERR_UNSUPPORTED;
  if (c->residual_len % c->k_group != 0) return KVQ_ERR_INVALID_ARG;
  if (c->residual_len > kMaxResidual) return KVQ_ERR_UNSUPPORTED;
  if (c->gqa_ratio > kMaxGqa) return KVQ_ERR_UNSUPPORTED;
  if (c->n_kv_heads > 255 || c->batch > 4095 || c->max_seq_len > (1 << 24)) return KVQ_ERR_UNSUPPORTED;
  if (c->symmetric != 0 && c->symmetric != 1) return KVQ_ERR_INVALID_ARG;
  if (c->symmetric && (c->bits != 8 || vbits != 8 || c->v_group != c->d_head)) return KVQ_ERR_UNSUPPORTED;
  if (c->symmetric && c->residual_len != 0) return KVQ_ERR_INVALID_ARG;  // no residual window
  if (c->k_outliers < 0 || c->k_outliers > 4) return KVQ_ERR_UNSUPPORTED;
  // isolated key entries with per-channel keys: decode kernels for r <= 4 only
  if (c->k_outliers > 0 && !c->symmetric && c->gqa_ratio > 4) return KVQ_ERR_UNSUPPORTED;
  Geometry x;
  x.L = c->n_layers;
  x.B = c->batch;
  x.H = c->n_kv_heads;
  x.r = c->gqa_ratio;
  x.d = c->d_head;
  x.S_max = c->max_seq_len;
  x.bits = c->bits;
  x.vbits = vbits;
  x.G = c->k_group;
  x.Gv = c->v_group;
  x.R = c->residual_len;
  x.sym = c->symmetric;
  x.kout = c->k_outliers;
  x.R_eff = x.sym ? 1 : (c->residual_len > 0 ? c->residual_len : c->k_group);  // symmetric: Tq = T
  x.S_pad = ((int64_t)c->max_seq_len + kSeqAlign - 1) / kSeqAlign * kSeqAlign;
  x.rowK = (int64_t)x.d * x.bits / 8;
  x.rowV = (int64_t)x.d * x.vbits / 8;
  x.n_vg = x.d / x.Gv;
  x.k_codes_slice = x.S_pad * x.rowK;
  // group (scale, zero point) pairs or per-token scales, then kout entries per token
  x.k_meta_slice = (x.sym ? x.S_pad * 2 : (x.S_pad / x.G) * x.d * 4) + x.S_pad * x.kout * 4;
  x.k_resid_slice = x.sym ? 0 : (int64_t)x.R_eff * x.d * 2;
  x.v_codes_slice = x.S_pad * x.rowV;
  x.v_meta_slice = x.S_pad * x.n_vg * 4;
  x.n_slices = (int64_t)x.L * x.B * x.H;
  *g = x;
  return KVQ_OK;
}

// Tokens whose keys are quantized when T tokens are cached.
inline int64_t quantized_keys(const Geometry& g, int64_t T) { return (T / g.R_eff) * g.R_eff; }

// Decode split-K bound that does not depend on the device: the workspace is sized for it.
inline int64_t max_splits(const Geometry& g, int64_t T) {
  int64_t by_len = (T + 63) / 64;
  int64_t units = (int64_t)g.B * g.H;
  int64_t by_units = (2048 + units - 1) / units;
  int64_t m = by_len < by_units ? by_len : by_units;
  if (m > 256) m = 256;
  return m < 1 ? 1 : m;
}

// Workspace layout: error word (u32) at offset 0, tickets [B*H] u32 at 256, then
// (m, l) float2 [B][n_q][cap], then o float [B][n_q][cap][d].
struct WorkspaceLayout {
  int64_t cap;
  size_t err_off, tickets_off, ml_off, o_off, total;
};

inline WorkspaceLayout workspace_layout(const Geometry& g, int64_t T) {
  WorkspaceLayout w;
  w.cap = max_splits(g, T);
  const int64_t nq = (int64_t)g.H * g.r;
  auto up = [](size_t v) { return (v + 255) / 256 * 256; };
  w.err_off = 0;
  w.tickets_off = 256;
  w.ml_off = w.tickets_off + up((size_t)g.B * g.H * 4);
  w.o_off = w.ml_off + up((size_t)g.B * nq * w.cap * 8);
  w.total = w.o_off + up((size_t)g.B * nq * w.cap * g.d * 4);
  return w;
}

}  // namespace kvq
