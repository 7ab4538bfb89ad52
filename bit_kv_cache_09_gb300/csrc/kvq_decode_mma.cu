// kvq_decode_mma.cu — code-width dispatch of the tensor-core decode attention
// (kernels in kvq_decode_mma.cuh, one translation unit per key code width, and two for
// per-channel keys with isolated key entries).
#include "kvq_kernels.h"

namespace kvq {

cudaError_t launch_decode_mma_b8(const DecodeParams& p, int vbits, cudaStream_t stream);
cudaError_t launch_decode_mma_b4(const DecodeParams& p, int vbits, cudaStream_t stream);
cudaError_t launch_decode_mma_b2(const DecodeParams& p, int vbits, cudaStream_t stream);
int occupancy_decode_mma_b8(int r, int n_vg, int vbits);
int occupancy_decode_mma_b4(int r, int n_vg, int vbits);
int occupancy_decode_mma_b2(int r, int n_vg, int vbits);
int max_clusters_decode_mma_b8(int r, int n_vg, int cs, int nw, int vbits);
int max_clusters_decode_mma_b4(int r, int n_vg, int cs, int nw, int vbits);
int max_clusters_decode_mma_b2(int r, int n_vg, int cs, int nw, int vbits);
cudaError_t launch_decode_mma_sym(const DecodeParams& p, cudaStream_t stream);
cudaError_t launch_decode_mma_outl8(const DecodeParams& p, int vbits, cudaStream_t stream);
cudaError_t launch_decode_mma_outl42(const DecodeParams& p, int bits, cudaStream_t stream);
int occupancy_decode_mma_outl8(int n_vg, int vbits);
int occupancy_decode_mma_outl42(int n_vg, int bits);
int max_clusters_decode_mma_outl8(int n_vg, int cs, int nw, int vbits);
int max_clusters_decode_mma_outl42(int n_vg, int cs, int nw, int bits);
int occupancy_decode_mma_sym(int r, int outl);
int max_clusters_decode_mma_sym(int r, int cs, int nw, int outl);

cudaError_t launch_decode_mma(const DecodeParams& p, int bits, int vbits, cudaStream_t stream) {
  if (p.sym) return launch_decode_mma_sym(p, stream);
  if (p.kout > 0) return bits == 8 ? launch_decode_mma_outl8(p, vbits, stream) : launch_decode_mma_outl42(p, bits, stream);
  switch (bits) {
    case 8: return launch_decode_mma_b8(p, vbits, stream);
    case 4: return launch_decode_mma_b4(p, vbits, stream);
    default: return launch_decode_mma_b2(p, vbits, stream);
  }
}

int occupancy_decode_mma(int bits, int vbits, int r, int n_vg, int sym) {
  if (sym == 3) return bits == 8 ? occupancy_decode_mma_outl8(n_vg, vbits) : occupancy_decode_mma_outl42(n_vg, bits);
  if (sym) return occupancy_decode_mma_sym(r, sym > 1);
  switch (bits) {
    case 8: return occupancy_decode_mma_b8(r, n_vg, vbits);
    case 4: return occupancy_decode_mma_b4(r, n_vg, vbits);
    default: return occupancy_decode_mma_b2(r, n_vg, vbits);
  }
}

int max_clusters_decode_mma(int bits, int vbits, int r, int n_vg, int cs, int nw, int sym) {
  if (sym == 3)
    return bits == 8 ? max_clusters_decode_mma_outl8(n_vg, cs, nw, vbits) : max_clusters_decode_mma_outl42(n_vg, cs, nw, bits);
  if (sym) return max_clusters_decode_mma_sym(r, cs, nw, sym > 1);
  switch (bits) {
    case 8: return max_clusters_decode_mma_b8(r, n_vg, cs, nw, vbits);
    case 4: return max_clusters_decode_mma_b4(r, n_vg, cs, nw, vbits);
    default: return max_clusters_decode_mma_b2(r, n_vg, cs, nw, vbits);
  }
}

}  // namespace kvq
