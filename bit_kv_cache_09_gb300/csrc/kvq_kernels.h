// kvq_kernels.h — kernel parameter blocks and launchers (library-internal).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "../../include/kvq.h"

namespace kvq {

// All pointers are already offset to the layer's first slice (layer, batch 0, head 0).
// Division by an invariant 32-bit divisor d of dividends below 2^31 (Granlund and
// Montgomery, "Division by invariant integers using multiplication", PLDI 1994):
// with l = ceil(log2 d), mul = ceil(2^(31+l) / d) < 2^32 and x < 2^31,
// floor(x / d) = umulhi(x, mul) >> (l - 1) (the excess of mul*d over 2^(31+l) is below d,
// so it moves x*mul / 2^(31+l) above x/d by less than 1/d). mul = 0 encodes d = 1.
struct FastDiv {
  uint32_t mul, shift;
};

inline FastDiv make_fast_div(uint32_t d) {
  FastDiv f{0u, 0u};
  if (d <= 1) return f;
  uint32_t l = 0;
  while ((1ull << l) < d) ++l;
  f.mul = (uint32_t)(((1ull << (31 + l)) + d - 1) / d);
  f.shift = l - 1;
  return f;
}

#ifdef __CUDACC__
__device__ __forceinline__ uint32_t fast_div(uint32_t x, FastDiv f) {
  return f.mul ? (__umulhi(x, f.mul) >> f.shift) : x;
}
#endif

struct AppendParams {
  uint8_t* k_codes;
  __half2* k_meta;
  __half* k_resid;
  uint8_t* v_codes;
  __half2* v_meta;
  const __half* k_in;  // [B][n_new][H][d]
  const __half* v_in;  // [B][n_new][H][d]
  int64_t s_cur, n_new;
  int64_t A1;      // first token of the residual window after the call
  int64_t group0;  // first key group quantized by this call
  int n_groups;    // key groups quantized by this call
  int B, H, G, Gv, R_eff, n_vg;
  int64_t S_pad, rowK, rowV;
  int64_t k_codes_slice, v_codes_slice;
  int64_t k_meta_slice;  // bytes of k_meta per slice
  FastDiv fd_H;     // division by H of value-row indices below 2^31
  int rows_32;      // n_new * H < 2^31: value-row indices fit the fast division
  int sym;          // symmetric per-token int8 scheme (k_meta: one binary16 scale per token)
  int kout;         // isolated key entries per token (after the key scales or group metadata)
  int wide_keys;    // key groups of 64/128 tokens on 16-warp CTAs (isolated key entries); else 8
};

struct DequantParams {
  const uint8_t* k_codes;
  const __half2* k_meta;
  const __half* k_resid;
  const uint8_t* v_codes;
  const __half2* v_meta;
  float* k_out;  // [B][H][T][d]
  float* v_out;
  int64_t T, Tq;
  int B, H, G, Gv, R_eff, n_vg;
  int64_t S_pad, rowK, rowV;
  int64_t k_codes_slice, v_codes_slice;
  int64_t k_meta_slice;  // bytes of k_meta per slice
  int sym;  // symmetric per-token int8 scheme (k_meta: one binary16 scale per token)
  int kout;  // isolated key entries per token (after the key scales or group metadata)
};

struct DecodeParams {
  const uint8_t* k_codes;
  const __half2* k_meta;
  const __half* k_resid;
  const uint8_t* v_codes;
  const __half2* v_meta;
  const __half* q;  // [B][H*r][d]
  // fused decode step (tensor-core kernel only): when k_new/v_new are set, the CTA that
  // owns token T-1 first appends it (value quantized per group, key into the residual)
  const __half* k_new;  // [B][1][H][d] or null
  const __half* v_new;  // [B][1][H][d] or null
  __half* k_resid_w;
  uint8_t* v_codes_w;
  __half2* v_meta_w;
  uint8_t* k_codes_w;  // symmetric scheme: the new key row is quantized in place
  __half2* k_meta_w;
  float* out;       // [B][H*r][d]
  uint32_t* err;      // error word (KVQ_DECODE_ERR_* bits), read by kvq_decode_error
  uint64_t wait_ns;   // time limit of every bounded wait of the tensor-core kernel (0: give up at once)
  uint32_t* tickets;  // [B*H]
  float2* ws_ml;      // [B][H*r][cap] (running max in log2 units, denominator)
  float* ws_o;        // [B][H*r][cap][d]
  int64_t T, Tq;
  int64_t chunk;      // tokens per split (multiple of 128)
  int n_split, cap;
  // mixed plan (tensor-core kernel, no clusters): a one-dimensional grid where the first
  // pairs_hi (batch row, kv head) pairs take n_hi splits of chunk_hi tokens and the other
  // pairs n_hi - 1 splits of chunk_lo tokens (pairs in slice order); 0: grid (n_split, H, B)
  int mixed;
  int n_hi, pairs_hi;
  int64_t chunk_hi, chunk_lo;
  int cluster;        // CTAs per cluster (splits merged through distributed shared memory)
  int warps;          // warps per CTA of the tensor-core kernel: 4, or 8 (cluster merges only)
  int n_parts;        // partials merged through the workspace: n_split / cluster
  int sym;            // symmetric per-token int8 scheme (k_meta: one binary16 scale per token)
  int kout;           // isolated key entries per token (after the key scales or group metadata)
  int early;          // tensor-core kernel: the first stages are copied before the wait on the
                      // previous kernel of the stream (the caller guarantees it writes no cache
                      // memory of this layer); queries and new rows are read after the wait
  int B, H, r, G, Gv, R_eff, n_vg;
  int log2G;          // G is a power of two
  int64_t S_pad, rowK, rowV;
  int64_t k_codes_slice, v_codes_slice;
  int64_t k_meta_slice;  // bytes of k_meta per slice
  float scale_log2;   // softmax_scale * log2(e)
};

// Programmatic dependent launch: a kernel launched with the attribute may start while
// the previous kernel of the stream finishes; it runs pdl_wait() before touching any
// global memory, which blocks until that kernel has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_allow_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Time limit of the tensor-core kernel's bounded waits unless a call asks for 0.
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

// One checked decode-attention launch (kvq_api.cu): decode_prepare validates every
// argument and fills it without touching the device; decode_enqueue launches it.
struct DecodeCall {
  DecodeParams p;
  bool simt;
  int bits, vbits;
  size_t counters_bytes;  // leading workspace bytes (error word, tickets) that must start at zero
};

// bits, vbits: key and value code widths (equal, or 8 and 4)
cudaError_t launch_append(const AppendParams& p, int bits, int vbits, cudaStream_t stream);
cudaError_t launch_dequant(const DequantParams& p, int bits, int vbits, cudaStream_t stream);
cudaError_t launch_decode_simt(const DecodeParams& p, int bits, cudaStream_t stream);  // equal widths only
cudaError_t launch_decode_mma(const DecodeParams& p, int bits, int vbits, cudaStream_t stream);
// sym: 0 asymmetric; 1 the symmetric per-token int8 scheme (bits == vbits == 8, n_vg == 1);
// 2 the symmetric scheme with isolated key entries; 3 asymmetric with isolated key entries (r <= 4)
int occupancy_decode_mma(int bits, int vbits, int r, int n_vg, int sym);  // resident CTAs per SM (0 on error)
int max_clusters_decode_mma(int bits, int vbits, int r, int n_vg, int cs, int nw, int sym);  // resident clusters of cs CTAs
int occupancy_decode_simt(int bits);

kvq_status decode_prepare(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                          const void* q_f16, float softmax_scale, float* out, void* ws, size_t ws_bytes,
                          kvq_decode_impl impl, const void* k_new, const void* v_new, bool early, uint64_t wait_ns,
                          DecodeCall* call);
kvq_status decode_enqueue(const DecodeCall& call, cudaStream_t stream);
kvq_status read_error_word(uint32_t* err, cudaStream_t stream, uint32_t* out);

}  // namespace kvq
