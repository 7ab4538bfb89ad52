// kvq_decode_mma.cu — bit-width dispatch of the tensor-core decode attention
// (kernels in kvq_decode_mma.cuh, one translation unit per code width).
#include "kvq_kernels.h"

namespace kvq {

cudaError_t launch_decode_mma_b8(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_mma_b4(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_mma_b2(const DecodeParams& p, cudaStream_t stream);
int occupancy_decode_mma_b8(int r, int n_vg);
int occupancy_decode_mma_b4(int r, int n_vg);
int occupancy_decode_mma_b2(int r, int n_vg);
int max_clusters_decode_mma_b8(int r, int n_vg, int cs, int nw);
int max_clusters_decode_mma_b4(int r, int n_vg, int cs, int nw);
int max_clusters_decode_mma_b2(int r, int n_vg, int cs, int nw);

cudaError_t launch_decode_mma(const DecodeParams& p, int bits, cudaStream_t stream) {
  switch (bits) {
    case 8: return launch_decode_mma_b8(p, stream);
    case 4: return launch_decode_mma_b4(p, stream);
    default: return launch_decode_mma_b2(p, stream);
  }
}

int occupancy_decode_mma(int bits, int r, int n_vg) {
  switch (bits) {
    case 8: return occupancy_decode_mma_b8(r, n_vg);
    case 4: return occupancy_decode_mma_b4(r, n_vg);
    default: return occupancy_decode_mma_b2(r, n_vg);
  }
}

int max_clusters_decode_mma(int bits, int r, int n_vg, int cs, int nw) {
  switch (bits) {
    case 8: return max_clusters_decode_mma_b8(r, n_vg, cs, nw);
    case 4: return max_clusters_decode_mma_b4(r, n_vg, cs, nw);
    default: return max_clusters_decode_mma_b2(r, n_vg, cs, nw);
  }
}

}  // namespace kvq
