// kvq_decode_mma_outl8.cu — instantiations of the tensor-core decode attention for
// per-channel keys with isolated key entries (OUTL), 8-bit keys (8- or 4-bit values), r <= 4.
#include "kvq_decode_mma_outl.cuh"

namespace kvq {

cudaError_t launch_decode_mma_outl8(const DecodeParams& p, int vbits, cudaStream_t stream) {
  return vbits == 4 ? mma::launch_outl_bits<8, 4>(p, stream) : mma::launch_outl_bits<8, 8>(p, stream);
}

int occupancy_decode_mma_outl8(int n_vg, int vbits) {
  return vbits == 4 ? mma::occupancy_outl_bits<8, 4>(n_vg) : mma::occupancy_outl_bits<8, 8>(n_vg);
}

int max_clusters_decode_mma_outl8(int n_vg, int cs, int nw, int vbits) {
  return vbits == 4 ? mma::max_clusters_outl_bits<8, 4>(n_vg, cs, nw) : mma::max_clusters_outl_bits<8, 8>(n_vg, cs, nw);
}

}  // namespace kvq
