// kvq_decode_mma_b8.cu — instantiations of the tensor-core decode attention for 8-bit
// key codes (with 8-bit values, or 4-bit values: the mixed-width configuration).
#include "kvq_decode_mma.cuh"

namespace kvq {

cudaError_t launch_decode_mma_b8(const DecodeParams& p, int vbits, cudaStream_t stream) {
  return vbits == 4 ? mma::launch_bits<8, 4>(p, stream) : mma::launch_bits<8, 8>(p, stream);
}

int occupancy_decode_mma_b8(int r, int n_vg, int vbits) {
  return vbits == 4 ? mma::occupancy_bits<8, 4>(r, n_vg) : mma::occupancy_bits<8, 8>(r, n_vg);
}

int max_clusters_decode_mma_b8(int r, int n_vg, int cs, int nw, int vbits) {
  return vbits == 4 ? mma::max_clusters_bits<8, 4>(r, n_vg, cs, nw) : mma::max_clusters_bits<8, 8>(r, n_vg, cs, nw);
}

}  // namespace kvq
