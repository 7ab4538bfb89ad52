// kvq_decode_mma_outl42.cu — instantiations of the tensor-core decode attention for
// per-channel keys with isolated key entries (OUTL), 4- and 2-bit codes, r <= 4.
#include "kvq_decode_mma_outl.cuh"

namespace kvq {

cudaError_t launch_decode_mma_outl42(const DecodeParams& p, int bits, cudaStream_t stream) {
  return bits == 4 ? mma::launch_outl_bits<4, 4>(p, stream) : mma::launch_outl_bits<2, 2>(p, stream);
}

int occupancy_decode_mma_outl42(int n_vg, int bits) {
  return bits == 4 ? mma::occupancy_outl_bits<4, 4>(n_vg) : mma::occupancy_outl_bits<2, 2>(n_vg);
}

int max_clusters_decode_mma_outl42(int n_vg, int cs, int nw, int bits) {
  return bits == 4 ? mma::max_clusters_outl_bits<4, 4>(n_vg, cs, nw) : mma::max_clusters_outl_bits<2, 2>(n_vg, cs, nw);
}

}  // namespace kvq
