// kvq_decode_mma_sym.cu — instantiations of the tensor-core decode attention for the
// symmetric per-token int8 scheme (8-bit keys and values, one value group, zero point 0),
// without and with isolated key entries (OUTL: the sparse side list read per score).
#include "kvq_decode_mma.cuh"

namespace kvq {

namespace {

template <bool OUTL>
cudaError_t launch_sym(const DecodeParams& p, cudaStream_t stream) {
  if (p.warps == 8 || p.warps == 5) {
    if (p.n_parts != 1) return cudaErrorInvalidConfiguration;  // 5- and 8-warp CTAs merge in clusters only
    if (p.warps == 5)
      return p.r <= 4 ? mma::launch_cfg<8, 8, 1, 1, 5, true, OUTL>(p, stream)
                      : mma::launch_cfg<8, 8, 2, 1, 5, true, OUTL>(p, stream);
    return p.r <= 4 ? mma::launch_cfg<8, 8, 1, 1, 8, true, OUTL>(p, stream)
                    : mma::launch_cfg<8, 8, 2, 1, 8, true, OUTL>(p, stream);
  }
  return p.r <= 4 ? mma::launch_cfg<8, 8, 1, 1, 4, true, OUTL>(p, stream)
                  : mma::launch_cfg<8, 8, 2, 1, 4, true, OUTL>(p, stream);
}

template <bool OUTL>
int max_clusters_sym(int r, int cs, int nw) {
  if (nw == 5)
    return r <= 4 ? mma::max_clusters_cfg<8, 8, 1, 1, 5, true, OUTL>(cs) : mma::max_clusters_cfg<8, 8, 2, 1, 5, true, OUTL>(cs);
  if (nw == 8)
    return r <= 4 ? mma::max_clusters_cfg<8, 8, 1, 1, 8, true, OUTL>(cs) : mma::max_clusters_cfg<8, 8, 2, 1, 8, true, OUTL>(cs);
  return r <= 4 ? mma::max_clusters_cfg<8, 8, 1, 1, 4, true, OUTL>(cs) : mma::max_clusters_cfg<8, 8, 2, 1, 4, true, OUTL>(cs);
}

}  // namespace

cudaError_t launch_decode_mma_sym(const DecodeParams& p, cudaStream_t stream) {
  if (p.n_vg != 1 || p.kout < 0 || p.kout > 4) return cudaErrorInvalidConfiguration;
  return p.kout > 0 ? launch_sym<true>(p, stream) : launch_sym<false>(p, stream);
}

int occupancy_decode_mma_sym(int r, int outl) {
  if (outl) return r <= 4 ? mma::occupancy_cfg<8, 8, 1, 1, true, true>() : mma::occupancy_cfg<8, 8, 2, 1, true, true>();
  return r <= 4 ? mma::occupancy_cfg<8, 8, 1, 1, true>() : mma::occupancy_cfg<8, 8, 2, 1, true>();
}

int max_clusters_decode_mma_sym(int r, int cs, int nw, int outl) {
  return outl ? max_clusters_sym<true>(r, cs, nw) : max_clusters_sym<false>(r, cs, nw);
}

}  // namespace kvq
