// kvq_decode_mma_outl.cuh — dispatch of the tensor-core decode attention for per-channel
// keys with isolated key entries (OUTL): r <= 4 (one query per score column pair),
// every value-group count and CTA width (library-internal).
#pragma once

#include "kvq_decode_mma.cuh"

namespace kvq {
namespace mma {

template <int BITS, int VBITS, int NW>
cudaError_t launch_outl_nw(const DecodeParams& p, cudaStream_t stream) {
  if (p.n_vg == 1) return launch_cfg<BITS, VBITS, 1, 1, NW, false, true>(p, stream);
  if (p.n_vg == 2) return launch_cfg<BITS, VBITS, 1, 2, NW, false, true>(p, stream);
  return launch_cfg<BITS, VBITS, 1, 4, NW, false, true>(p, stream);
}

template <int BITS, int VBITS>
cudaError_t launch_outl_bits(const DecodeParams& p, cudaStream_t stream) {
  if (p.r > 4 || p.kout < 1 || p.kout > 4) return cudaErrorInvalidConfiguration;
  if (p.warps == 8 || p.warps == 5) {
    if (p.n_parts != 1) return cudaErrorInvalidConfiguration;  // 5- and 8-warp CTAs merge in clusters only
    return p.warps == 8 ? launch_outl_nw<BITS, VBITS, 8>(p, stream) : launch_outl_nw<BITS, VBITS, 5>(p, stream);
  }
  return launch_outl_nw<BITS, VBITS, 4>(p, stream);
}

template <int BITS, int VBITS>
int occupancy_outl_bits(int n_vg) {
  if (n_vg == 1) return occupancy_cfg<BITS, VBITS, 1, 1, false, true>();
  if (n_vg == 2) return occupancy_cfg<BITS, VBITS, 1, 2, false, true>();
  return occupancy_cfg<BITS, VBITS, 1, 4, false, true>();
}

template <int BITS, int VBITS, int NW>
int max_clusters_outl_nw(int n_vg, int cs) {
  if (n_vg == 1) return max_clusters_cfg<BITS, VBITS, 1, 1, NW, false, true>(cs);
  if (n_vg == 2) return max_clusters_cfg<BITS, VBITS, 1, 2, NW, false, true>(cs);
  return max_clusters_cfg<BITS, VBITS, 1, 4, NW, false, true>(cs);
}

template <int BITS, int VBITS>
int max_clusters_outl_bits(int n_vg, int cs, int nw) {
  if (nw == 5) return max_clusters_outl_nw<BITS, VBITS, 5>(n_vg, cs);
  return nw == 8 ? max_clusters_outl_nw<BITS, VBITS, 8>(n_vg, cs) : max_clusters_outl_nw<BITS, VBITS, 4>(n_vg, cs);
}

}  // namespace mma
}  // namespace kvq
