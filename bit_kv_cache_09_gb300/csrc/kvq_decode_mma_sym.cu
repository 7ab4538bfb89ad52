// kvq_decode_mma_sym.cu — instantiations of the tensor-core decode attention for the
// symmetric per-token int8 scheme (8-bit keys and values, one value group, zero point 0).
#include "kvq_decode_mma.cuh"

namespace kvq {

cudaError_t launch_decode_mma_sym(const DecodeParams& p, cudaStream_t stream) {
  if (p.n_vg != 1) return cudaErrorInvalidConfiguration;
  if (p.warps == 8 || p.warps == 5) {
    if (p.n_parts != 1) return cudaErrorInvalidConfiguration;  // 5- and 8-warp CTAs merge in clusters only
    if (p.warps == 5)
      return p.r <= 4 ? mma::launch_cfg<8, 8, 1, 1, 5, true>(p, stream) : mma::launch_cfg<8, 8, 2, 1, 5, true>(p, stream);
    return p.r <= 4 ? mma::launch_cfg<8, 8, 1, 1, 8, true>(p, stream) : mma::launch_cfg<8, 8, 2, 1, 8, true>(p, stream);
  }
  return p.r <= 4 ? mma::launch_cfg<8, 8, 1, 1, 4, true>(p, stream) : mma::launch_cfg<8, 8, 2, 1, 4, true>(p, stream);
}

int occupancy_decode_mma_sym(int r) {
  return r <= 4 ? mma::occupancy_cfg<8, 8, 1, 1, true>() : mma::occupancy_cfg<8, 8, 2, 1, true>();
}

int max_clusters_decode_mma_sym(int r, int cs, int nw) {
  if (nw == 5)
    return r <= 4 ? mma::max_clusters_cfg<8, 8, 1, 1, 5, true>(cs) : mma::max_clusters_cfg<8, 8, 2, 1, 5, true>(cs);
  if (nw == 8)
    return r <= 4 ? mma::max_clusters_cfg<8, 8, 1, 1, 8, true>(cs) : mma::max_clusters_cfg<8, 8, 2, 1, 8, true>(cs);
  return r <= 4 ? mma::max_clusters_cfg<8, 8, 1, 1, 4, true>(cs) : mma::max_clusters_cfg<8, 8, 2, 1, 4, true>(cs);
}

}  // namespace kvq
