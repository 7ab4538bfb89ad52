// kvq_noalloc.cu — decode attention whose split-K scratch lives in a static device
// array, for callers that cannot allocate device memory.
//
// kvq_decode_attention needs a workspace (split-K partials, per-(batch row, kv head)
// counters, an error word) that the caller allocates. Some callers cannot do that
// at the point of the call: code embedded in a host framework whose allocator owns
// all device memory and forbids raw cudaMalloc/cudaFree, code that runs where an
// allocation's implicit device synchronisation is not acceptable (a latency-critical
// decode loop), or code with no allocator handle at hand. This entry point serves
// them: the scratch is a file-scope __device__ array of kStaticScratchBytes, which
// every GPU that loads the library keeps until the process exits.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "kvq_common.cuh"
#include "kvq_kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scratch on the current device (looked up once per device).
cudaError_t scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

extern "C" kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer,
                                                   int64_t s_cur, const void* q_f16, float softmax_scale, float* out,
                                                   void* stream) {
  kvq::Geometry g;
  const kvq_status st = kvq::make_geometry(cfg, &g);
  if (st != KVQ_OK) return st;
  if (s_cur < 1) return KVQ_ERR_INVALID_ARG;
  if (kvq::workspace_layout(g, s_cur).total > kStaticScratchBytes) return KVQ_ERR_WORKSPACE;  // beyond the static scratch
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  // Every argument is checked before the shared array is touched: a rejected call
  // writes nothing into it (another stream's decode may be using it).
  kvq::DecodeCall call;
  const kvq_status chk = kvq::decode_prepare(cfg, bufs, layer, s_cur, q_f16, softmax_scale, out, scratch,
                                             kStaticScratchBytes, KVQ_DECODE_AUTO, nullptr, nullptr, false,
                                             kvq::kDefaultWaitNs, &call);
  if (chk != KVQ_OK) return chk;
  // The error word and the split counters must start at zero; the array keeps the
  // previous call's contents, so clear them on the caller's stream.
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, call.counters_bytes, s) != cudaSuccess) return KVQ_ERR_CUDA;
  return kvq::decode_enqueue(call, s);
}

extern "C" kvq_status kvq_decode_noalloc_error(void* stream, uint32_t* err_out) {
  if (!err_out) return KVQ_ERR_INVALID_ARG;
  void* scratch = nullptr;
  if (scratch_address(&scratch) != cudaSuccess) return KVQ_ERR_CUDA;
  return kvq::read_error_word(static_cast<uint32_t*>(scratch), static_cast<cudaStream_t>(stream), err_out);
}
