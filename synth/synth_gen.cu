// synth_gen.cu — device implementation of the seeded synthetic K / V / query
// generator defined in synth/__init__.py (splitmix64 counters, Irwin–Hall sums of
// twelve 16-bit uniforms). It holds none of the quantization or attention
// arithmetic; it only produces inputs, bit-identical to the host implementation.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

namespace {

constexpr uint64_t kGolden = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t mix64(uint64_t x) {
  x ^= x >> 30;
  x *= 0xBF58476D1CE4E5B9ull;
  x ^= x >> 27;
  x *= 0x94D049BB133111EBull;
  x ^= x >> 31;
  return x;
}

__device__ __forceinline__ uint64_t counter(uint64_t stream, uint64_t layer, uint64_t head, uint64_t ch, uint64_t b,
                                            uint64_t t) {
  return (stream << 60) | (layer << 52) | (head << 44) | (ch << 36) | (b << 24) | t;
}

__device__ __forceinline__ int64_t normal_m(uint64_t seed, uint64_t ctr) {
  const uint64_t base = mix64((seed * kGolden) ^ ctr);
  int64_t total = 0;
#pragma unroll
  for (int k = 1; k <= 3; ++k) {
    const uint64_t w = mix64(base + (uint64_t)k * kGolden);
    total += (int64_t)(w & 0xFFFF) + (int64_t)((w >> 16) & 0xFFFF) + (int64_t)((w >> 32) & 0xFFFF) +
             (int64_t)((w >> 48) & 0xFFFF);
  }
  return total - 6 * 65536;
}

// out[b][t][h][c], stream 0 = keys (outlier channels: gain * m + shift65536), 1 = values.
__global__ void gen_kv_kernel(uint64_t seed, int stream_kind, int layer, int b0, int64_t t0, int64_t nt, int H, int d,
                              const uint64_t* __restrict__ outlier_words, int gain, int64_t shift65536, __half* out,
                              int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  const int wpr = (d + 63) / 64;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int c = (int)(i % d);
    int64_t r = i / d;
    const int h = (int)(r % H);
    r /= H;
    const int64_t t = t0 + r % nt;
    const int b = b0 + (int)(r / nt);
    const int64_t m = normal_m(seed, counter((uint64_t)stream_kind, layer, h, c, b, t));
    float v;
    if (stream_kind == 1) {
      v = (float)m * 7.62939453125e-06f;  // 2^-17, exact
    } else {
      const bool outlier = outlier_words && ((outlier_words[h * wpr + c / 64] >> (c % 64)) & 1ull);
      if (outlier) v = __ll2float_rn(m * gain + shift65536) * 1.52587890625e-05f;  // * 2^-16, exact
      else v = (float)m * 1.52587890625e-05f;
    }
    out[i] = __float2half_rn(v);
  }
}

// q[b][i][c] for the decode step at token index step_token.
__global__ void gen_q_kernel(uint64_t seed, int layer, int b0, int n_q, int d, int64_t step_token, __half* out,
                             int64_t n) {
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
    const int c = (int)(i % d);
    const int64_t r = i / d;
    const int qh = (int)(r % n_q);
    const int b = b0 + (int)(r / n_q);
    const int64_t m = normal_m(seed, counter(2, layer, qh, c, b, step_token));
    out[i] = __float2half_rn((float)m * 1.52587890625e-05f);
  }
}

}  // namespace

extern "C" {

// Keys (stream_kind 0) or values (1) of batch rows [b0, b0+nb) and tokens [t0, t0+nt):
// out [nb][nt][H][d] binary16 (device). outlier_words: device [H][ceil(d/64)] bit masks
// (keys only; may be null). Returns a cudaError_t value.
int synth_gen_kv(uint64_t seed, int stream_kind, int layer, int b0, int nb, int64_t t0, int64_t nt, int H, int d,
                 const void* outlier_words, int gain, int64_t shift65536, void* out, void* stream) {
  const int64_t n = (int64_t)nb * nt * H * d;
  if (n <= 0) return 0;
  const int64_t blocks64 = (n + 255) / 256;
  const int blocks = (int)(blocks64 < 65536 ? blocks64 : 65536);
  gen_kv_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      seed, stream_kind, layer, b0, t0, nt, H, d, static_cast<const uint64_t*>(outlier_words), gain, shift65536,
      static_cast<__half*>(out), n);
  return (int)cudaGetLastError();
}

int synth_gen_q(uint64_t seed, int layer, int b0, int nb, int n_q, int d, int64_t step_token, void* out, void* stream) {
  const int64_t n = (int64_t)nb * n_q * d;
  if (n <= 0) return 0;
  const int64_t blocks64 = (n + 255) / 256;
  const int blocks = (int)(blocks64 < 65536 ? blocks64 : 65536);
  gen_q_kernel<<<blocks, 256, 0, static_cast<cudaStream_t>(stream)>>>(seed, layer, b0, n_q, d, step_token,
                                                                      static_cast<__half*>(out), n);
  return (int)cudaGetLastError();
}

}  // extern "C"
