// kvq_decode_simt.cu — split-K decode attention on the CUDA cores (binary32 FMA).
//
// Reads the packed integer cache and dequantizes on the fly ("KV Cache Quantization —
// 8-bit and 4-bit", § Decode is memory-bound, so smaller is also faster), with the
// key scales running along channels and the value scales along tokens inside one
// loop ("Sub-8-Bit KV Cache Quantization Is Not a Free Lever for an RDNA4 Agent
// Swarm", § The RDNA4 kernel angle). Per key group the channel scales fold into the
// query: q . k_hat = sum_c (q_c s_c) u_c + sum_c q_c s_c (q_min - zp_c).
//
// One CTA per (split, kv head, batch row), 128 threads, tiles of 128 tokens:
//   phase 1: thread = token, r scores (log2 units);
//   phase 2: warp = query head, online-softmax update (running max m, sum l);
//   phase 3: thread = channel, o[i] = alpha_i * o[i] + sum_t p_it * v_hat_tc.
// Splits write (m, l, o) partials; the last CTA of a (batch row, kv head) to finish
// (atomic ticket, no waiting) merges them with log-sum-exp weights.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq_common.cuh"
#include "kvq_kernels.h"
#include "kvq_merge.cuh"

namespace kvq {
namespace {

constexpr int kTile = 128;
constexpr int kRM = kMaxGqa;  // 8 query heads per CTA at most

template <int BITS>
__global__ void __launch_bounds__(128) decode_simt_kernel(DecodeParams p) {
  constexpr float qmin = -(float)(1 << (BITS - 1));
  constexpr int MASK = (1 << BITS) - 1;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t slice = (int64_t)b * p.H + h;
  const int nq = p.H * p.r;
  const int64_t t_begin = (int64_t)split * p.chunk;
  const int64_t t_end = min(t_begin + p.chunk, p.T);

  __shared__ __align__(16) float q_s[kHeadDim][kRM];         // raw query, [c][i]
  __shared__ __align__(16) float qk_s[4][kHeadDim][kRM];     // query * key scale per group in the tile
  __shared__ float biasp_s[4][4][kRM];                       // per-warp partial biases
  __shared__ float bias_s[4][kRM];
  __shared__ __align__(16) float sc_s[kTile][kRM];           // scores, then probabilities
  __shared__ __align__(16) uint32_t v_s[kTile * kHeadDim * BITS / 8 / 4];  // value pair rows of the tile
  __shared__ __half2 vm_s[kTile * 4];                        // value metadata of the tile
  __shared__ float m_s[kRM], l_s[kRM], a_s[kRM];

  // query of the r heads of this kv head (zero for unused heads)
  for (int idx = tid; idx < kHeadDim * kRM; idx += blockDim.x) {
    const int c = idx / kRM, i = idx % kRM;
    q_s[c][i] = (i < p.r) ? __half2float(p.q[((int64_t)b * nq + h * p.r + i) * kHeadDim + c]) : 0.0f;
  }
  if (tid < kRM) {
    m_s[tid] = -__int_as_float(0x7f800000);
    l_s[tid] = 0.0f;
  }
  float o[kRM];
#pragma unroll
  for (int i = 0; i < kRM; ++i) o[i] = 0.0f;

  const uint8_t* kc = p.k_codes + slice * p.k_codes_slice;
  const __half2* km = reinterpret_cast<const __half2*>(reinterpret_cast<const uint8_t*>(p.k_meta) + slice * p.k_meta_slice);
  const __half* kr = p.k_resid + slice * (int64_t)p.R_eff * kHeadDim;
  const uint8_t* vc = p.v_codes + slice * p.v_codes_slice;
  const __half2* vm = p.v_meta + slice * p.S_pad * p.n_vg;
  const int c_own = tid;  // channel owned in phase 3
  const int pos_own = 16 * (c_own & 7) + 2 * (c_own >> 4) + ((c_own >> 3) & 1);
  const int bit_own = pos_own * BITS;
  __syncthreads();

  for (int64_t t0 = t_begin; t0 < t_end; t0 += kTile) {
    const int n_valid = (int)min((int64_t)kTile, t_end - t0);
    // ---- phase 0: folded queries of the key groups in this tile, value tile to smem
    const int groups_in_tile = kTile / p.G;
    const int64_t g_first = t0 / p.G;
    for (int gi = 0; gi < groups_in_tile; ++gi) {
      const int64_t g = g_first + gi;
      if (g * p.G >= p.Tq) continue;  // residual tokens use the raw query
      const __half2 m = km[g * kHeadDim + c_own];
      const float s = __low2float(m), zofs = qmin - __high2float(m);
      float part[kRM];
#pragma unroll
      for (int i = 0; i < kRM; ++i) {
        const float qs = q_s[c_own][i] * s;
        qk_s[gi][c_own][i] = qs;
        part[i] = qs * zofs;
      }
#pragma unroll
      for (int i = 0; i < kRM; ++i) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) part[i] += __shfl_xor_sync(0xffffffffu, part[i], off);
      }
      if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kRM; ++i) biasp_s[gi][warp][i] = part[i];
      }
    }
    {
      const int words = kTile * kHeadDim * BITS / 8 / 4;
      const uint4* src = reinterpret_cast<const uint4*>(vc + (t0 >> 1) * 2 * p.rowV);
      for (int k = tid; k < words / 4; k += blockDim.x) reinterpret_cast<uint4*>(v_s)[k] = src[k];
      for (int k = tid; k < kTile * p.n_vg; k += blockDim.x) vm_s[k] = vm[t0 * p.n_vg + k];
    }
    __syncthreads();
    if (tid < 4 * kRM) {
      const int gi = tid / kRM, i = tid % kRM;
      bias_s[gi][i] = biasp_s[gi][0][i] + biasp_s[gi][1][i] + biasp_s[gi][2][i] + biasp_s[gi][3][i];
    }
    __syncthreads();

    // ---- phase 1: scores, thread = token
    {
      const int64_t t = t0 + tid;
      float acc[kRM];
#pragma unroll
      for (int i = 0; i < kRM; ++i) acc[i] = 0.0f;
      if (tid < n_valid) {
        if (t < p.Tq) {
          const int gi = (int)(t / p.G - g_first);
          const uint4* row = reinterpret_cast<const uint4*>(kc + t * p.rowK);
          constexpr int CHUNKS = kHeadDim * BITS / 128;  // 16-byte chunks per row
          constexpr int PER_WORD = 32 / BITS;
#pragma unroll
          for (int ch = 0; ch < CHUNKS; ++ch) {
            const uint4 w4 = row[ch];
            const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
#pragma unroll
              for (int e = 0; e < PER_WORD; ++e) {
                const int c = (ch * 4 + wi) * PER_WORD + e;
                const float u = (float)((ws[wi] >> (e * BITS)) & MASK);
                const float4 qa = *reinterpret_cast<const float4*>(&qk_s[gi][c][0]);
                const float4 qb = *reinterpret_cast<const float4*>(&qk_s[gi][c][4]);
                acc[0] += qa.x * u; acc[1] += qa.y * u; acc[2] += qa.z * u; acc[3] += qa.w * u;
                acc[4] += qb.x * u; acc[5] += qb.y * u; acc[6] += qb.z * u; acc[7] += qb.w * u;
              }
            }
          }
#pragma unroll
          for (int i = 0; i < kRM; ++i) acc[i] += bias_s[gi][i];
        } else {
          const uint4* row = reinterpret_cast<const uint4*>(kr + (t % p.R_eff) * kHeadDim);
#pragma unroll
          for (int ch = 0; ch < kHeadDim / 8; ++ch) {
            const uint4 w4 = row[ch];
            const uint32_t ws[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
            for (int wi = 0; wi < 4; ++wi) {
              const __half2 hv = *reinterpret_cast<const __half2*>(&ws[wi]);
              const float k0 = __low2float(hv), k1 = __high2float(hv);
              const int c = ch * 8 + wi * 2;
              const float4 qa0 = *reinterpret_cast<const float4*>(&q_s[c][0]);
              const float4 qb0 = *reinterpret_cast<const float4*>(&q_s[c][4]);
              const float4 qa1 = *reinterpret_cast<const float4*>(&q_s[c + 1][0]);
              const float4 qb1 = *reinterpret_cast<const float4*>(&q_s[c + 1][4]);
              acc[0] += qa0.x * k0 + qa1.x * k1; acc[1] += qa0.y * k0 + qa1.y * k1;
              acc[2] += qa0.z * k0 + qa1.z * k1; acc[3] += qa0.w * k0 + qa1.w * k1;
              acc[4] += qb0.x * k0 + qb1.x * k1; acc[5] += qb0.y * k0 + qb1.y * k1;
              acc[6] += qb0.z * k0 + qb1.z * k1; acc[7] += qb0.w * k0 + qb1.w * k1;
            }
          }
        }
#pragma unroll
        for (int i = 0; i < kRM; ++i) sc_s[tid][i] = acc[i] * p.scale_log2;
      } else {
#pragma unroll
        for (int i = 0; i < kRM; ++i) sc_s[tid][i] = -__int_as_float(0x7f800000);
      }
    }
    __syncthreads();

    // ---- phase 2: online softmax statistics, warp = query head
    for (int i = warp; i < p.r; i += 4) {
      float v[4];
      float mx = -__int_as_float(0x7f800000);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        v[k] = sc_s[lane + 32 * k][i];
        mx = fmaxf(mx, v[k]);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
      const float m_old = m_s[i];
      const float m_new = fmaxf(m_old, mx);
      float sum = 0.0f;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float pv = exp2f(v[k] - m_new);
        sc_s[lane + 32 * k][i] = pv;
        sum += pv;
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
      __syncwarp();
      if (lane == 0) {
        const float alpha = exp2f(m_old - m_new);
        a_s[i] = alpha;
        l_s[i] = l_s[i] * alpha + sum;
        m_s[i] = m_new;
      }
    }
    __syncthreads();

    // ---- phase 3: weighted values, thread = channel
    {
#pragma unroll
      for (int i = 0; i < kRM; ++i) o[i] *= (i < p.r) ? a_s[i] : 0.0f;
      const int words_per_pair = 2 * (int)p.rowV / 4;
      const int unit = bit_own >> 4, shift = bit_own & 15;
      const int vg = c_own / p.Gv;
      for (int tau = 0; tau < n_valid; ++tau) {
        const uint32_t word = v_s[(tau >> 1) * words_per_pair + unit];
        const uint32_t u = ((word >> (16 * (tau & 1))) >> shift) & MASK;
        // pair record {scale 2p, scale 2p+1, zp 2p, zp 2p+1} of group vg
        const __half* rec = reinterpret_cast<const __half*>(vm_s) + ((tau >> 1) * p.n_vg + vg) * 4 + (tau & 1);
        const float vh = __half2float(rec[0]) * ((float)u + qmin - __half2float(rec[2]));
        const float4 pa = *reinterpret_cast<const float4*>(&sc_s[tau][0]);
        const float4 pb = *reinterpret_cast<const float4*>(&sc_s[tau][4]);
        o[0] += pa.x * vh; o[1] += pa.y * vh; o[2] += pa.z * vh; o[3] += pa.w * vh;
        o[4] += pb.x * vh; o[5] += pb.y * vh; o[6] += pb.z * vh; o[7] += pb.w * vh;
      }
    }
    __syncthreads();
  }

  // ---- epilogue: direct output or split-K partial + last-CTA merge
  const int64_t qrow0 = (int64_t)b * nq + (int64_t)h * p.r;
  if (p.n_split == 1) {
    for (int i = 0; i < p.r; ++i) p.out[(qrow0 + i) * kHeadDim + c_own] = o[i] / l_s[i];
    return;
  }
  for (int i = 0; i < p.r; ++i) p.ws_o[((qrow0 + i) * p.cap + split) * kHeadDim + c_own] = o[i];
  if (tid < p.r) p.ws_ml[(qrow0 + tid) * p.cap + split] = make_float2(m_s[tid], l_s[tid]);
  merge_if_last(p, p.n_parts, slice, qrow0, &qk_s[0][0][0]);  // the folded-query buffer is free now
}

}  // namespace

int occupancy_decode_simt(int bits) {
  int n = 0;
  cudaError_t e = bits == 8 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<8>, 128, 0)
                  : bits == 4 ? cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<4>, 128, 0)
                              : cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_simt_kernel<2>, 128, 0);
  return e == cudaSuccess ? n : 0;
}

cudaError_t launch_decode_simt(const DecodeParams& p, int bits, cudaStream_t stream) {
  dim3 grid((unsigned)p.n_split, (unsigned)p.H, (unsigned)p.B);
  switch (bits) {
    case 8: decode_simt_kernel<8><<<grid, 128, 0, stream>>>(p); break;
    case 4: decode_simt_kernel<4><<<grid, 128, 0, stream>>>(p); break;
    default: decode_simt_kernel<2><<<grid, 128, 0, stream>>>(p); break;
  }
  return cudaGetLastError();
}

}  // namespace kvq
