// kvq_decode_mma_b4.cu — instantiations of the tensor-core decode attention for 4-bit codes.
#include "kvq_decode_mma.cuh"

namespace kvq {

cudaError_t launch_decode_mma_b4(const DecodeParams& p, int, cudaStream_t stream) {
  return mma::launch_bits<4, 4>(p, stream);
}

int occupancy_decode_mma_b4(int r, int n_vg, int) { return mma::occupancy_bits<4, 4>(r, n_vg); }

int max_clusters_decode_mma_b4(int r, int n_vg, int cs, int nw, int) {
  return mma::max_clusters_bits<4, 4>(r, n_vg, cs, nw);
}

}  // namespace kvq
