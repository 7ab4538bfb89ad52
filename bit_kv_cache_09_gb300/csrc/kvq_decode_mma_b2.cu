// kvq_decode_mma_b2.cu — instantiations of the tensor-core decode attention for 2-bit codes.
#include "kvq_decode_mma.cuh"

namespace kvq {

cudaError_t launch_decode_mma_b2(const DecodeParams& p, int, cudaStream_t stream) {
  return mma::launch_bits<2, 2>(p, stream);
}

int occupancy_decode_mma_b2(int r, int n_vg, int) { return mma::occupancy_bits<2, 2>(r, n_vg); }

int max_clusters_decode_mma_b2(int r, int n_vg, int cs, int nw, int) {
  return mma::max_clusters_bits<2, 2>(r, n_vg, cs, nw);
}

}  // namespace kvq
