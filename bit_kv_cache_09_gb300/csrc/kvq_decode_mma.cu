// kvq_decode_mma.cu — split-K decode attention with tensor-core products over the
// exact integer codes (mma.sync m16n8k16, binary16 operands, binary32 accumulation).
//
// Decode streams the whole packed cache once per step and reads integers that it
// dequantizes on the fly ("KV Cache Quantization — 8-bit and 4-bit", § Decode is
// memory-bound, so smaller is also faster); keys carry per-channel scales and values
// per-token scales inside the same loop ("Sub-8-Bit KV Cache Quantization Is Not a
// Free Lever for an RDNA4 Agent Swarm", § The RDNA4 kernel angle). With r = 4..8
// query heads per kv head the binary32 CUDA-core FMA work (2*r*d per token) exceeds
// what the FP32 pipe sustains at HBM speed for 4- and 2-bit codes, so both products
// run on the tensor cores:
//
//   scores  S[i][t] = sum_c (q_ic s_gc) u_tc + sum_c q_ic s_gc (q_min - zp_gc)
//           A = folded query (rows: query heads, hi and lo binary16 halves of a
//               per-row power-of-two-normalised binary32 value), B = key codes.
//   output  O[c][i] = sum_t u_tc (p_it s_tj) + sum_t p_it s_tj (q_min - zp_tj)
//           A = value codes (rows: channels), B = weights p*s (hi and lo halves).
//
// Codes enter the MMA as binary16 subnormals: the 16-bit pattern u IS the value
// u * 2^-24, so unpacking is a mask (and a byte permute for 8-bit codes), and the
// 2^24 factor is restored on the binary32 results. The zero-point sums are plain
// binary32 FMAs. Packed layouts are chosen so that every lane's fragment comes from
// one contiguous chunk (see include/kvq.h): key row chunk j of a lane holds channels
// [32j, 32j+32); value pair-row chunk g holds channels {16m + g, 16m + g + 8}.
//
// One CTA (4 warps) per (split, kv head, batch row); each warp owns a contiguous run
// of 16-token slabs with its own online softmax; the CTA merges its warps, and splits
// merge through the workspace (last CTA, atomic ticket, no waiting).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq_common.cuh"
#include "kvq_kernels.h"

namespace kvq {
namespace {

constexpr int kWarps = 4;
constexpr int kSlab = 16;

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0u), "r"(sel));
  return d;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// hi = binary16(x), lo = binary16(x - hi) for a pair, packed as half2 bit patterns.
__device__ __forceinline__ void split2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
  const __half2 h = __floats2half2_rn(x0, x1);
  const float2 hf = __half22float2(h);
  hi = h2_bits(h);
  lo = h2_bits(__floats2half2_rn(x0 - hf.x, x1 - hf.y));
}

// Words of one lane's chunk of a key row / value pair row.
template <int BITS>
struct Chunk {
  static constexpr int WORDS = BITS * 128 / 8 / 4 / 4;  // rowK/4 bytes in 32-bit words: 8, 4, 2
};

template <int BITS>
__device__ __forceinline__ void load_chunk(const uint8_t* p, uint32_t* w) {
  if (BITS == 8) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    const uint4 b = __ldg(reinterpret_cast<const uint4*>(p) + 1);
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else if (BITS == 4) {
    const uint4 a = __ldg(reinterpret_cast<const uint4*>(p));
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else {
    const uint2 a = __ldg(reinterpret_cast<const uint2*>(p));
    w[0] = a.x; w[1] = a.y;
  }
}

// Key codes: pair pi (0..15) of lane chunk j -> half2 of channels (ca, cb) as subnormals.
template <int BITS>
__device__ __forceinline__ uint32_t k_pair(const uint32_t* w, int pi) {
  if (BITS == 8) return prmt(w[pi >> 1], (pi & 1) ? 0x4342u : 0x4140u);
  if (BITS == 4) return (w[pi >> 2] >> (4 * (pi & 3))) & 0x000F000Fu;
  return (w[pi >> 3] >> (2 * (pi & 7))) & 0x00030003u;
}

// Local channel indices (within the lane's 32 channels) of key pair pi.
template <int BITS>
__device__ __forceinline__ int k_pair_ca(int pi) {
  if (BITS == 8) return 4 * (pi >> 1) + 2 * (pi & 1);
  if (BITS == 4) return 8 * (pi >> 2) + (pi & 3);
  return 16 * (pi >> 3) + (pi & 7);
}
template <int BITS>
__device__ __forceinline__ int k_pair_cb(int pi) {
  if (BITS == 8) return k_pair_ca<BITS>(pi) + 1;
  if (BITS == 4) return k_pair_ca<BITS>(pi) + 4;
  return k_pair_ca<BITS>(pi) + 8;
}

// Value codes: position i (0..15) of lane chunk g in a pair row -> half2(token 2p, token 2p+1).
template <int BITS>
__device__ __forceinline__ uint32_t v_pair(const uint32_t* w, int i) {
  if (BITS == 8) return prmt(w[i >> 1], (i & 1) ? 0x4341u : 0x4240u);
  if (BITS == 4) return (w[i >> 2] >> (4 * (i & 3))) & 0x000F000Fu;
  return (w[i >> 3] >> (2 * (i & 7))) & 0x00030003u;
}

template <int BITS, int NT>  // NT: PV n-tiles (1: r <= 4, hi/lo in one tile; 2: r <= 8, hi tile + lo tile)
__global__ void __launch_bounds__(kWarps * 32) decode_mma_kernel(DecodeParams p) {
  constexpr float qmin = -(float)(1 << (BITS - 1));
  constexpr int CW = Chunk<BITS>::WORDS;
  constexpr float kTwo24 = 16777216.0f;
  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, j = lane & 3;
  const int r = p.r;
  const int qi = (NT == 1) ? ((g & 3) % r) : (g % r);  // query head of QK row g / PV column g
  const bool lo_lane = (NT == 1) && (g >= 4);            // supplies the lo half of p in the PV tile
  const int64_t slice = (int64_t)b * p.H + h;
  const int nq = p.H * r;
  const int64_t qrow0 = (int64_t)b * nq + (int64_t)h * r;

  const int64_t t_begin = (int64_t)split * p.chunk;
  const int64_t t_end = min(t_begin + p.chunk, p.T);
  const int n_slabs = (int)((t_end - t_begin + kSlab - 1) / kSlab);
  const int spw = (n_slabs + kWarps - 1) / kWarps;
  const int slab0 = warp * spw;
  const int slab1 = min(n_slabs, slab0 + spw);

  const uint8_t* kc = p.k_codes + slice * p.k_codes_slice;
  const __half2* km = p.k_meta + slice * (p.S_pad / p.G) * kHeadDim;
  const __half* kr = p.k_resid + slice * (int64_t)p.R_eff * kHeadDim;
  const uint8_t* vc = p.v_codes + slice * p.v_codes_slice;
  const __half2* vm = p.v_meta + slice * p.S_pad * p.n_vg;

  // raw query of row qi, channels [32j, 32j+32), pre-scaled to log2 units
  float qf[32];
  {
    const uint4* qp = reinterpret_cast<const uint4*>(p.q + (qrow0 + qi) * kHeadDim + 32 * j);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const uint4 v = __ldg(qp + k);
      const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&ws[e]));
        qf[8 * k + 2 * e] = f.x;
        qf[8 * k + 2 * e + 1] = f.y;
      }
    }
  }

  // online softmax state of query qi (identical in the 4 lanes of row g)
  float m_run = -__int_as_float(0x7f800000), l_run = 0.0f;
  float o[8][NT][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int e = 0; e < 4; ++e) o[mt][nt][e] = 0.0f;
  float beta[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // zero-point sums per value group (n_vg <= 4)

  uint32_t qa[8][4];  // QK A fragments of the current key group (or of the raw query for residual keys)
  float qscale = 0.0f, qbias = 0.0f;
  int64_t cur_group = -1;

  for (int sl = slab0; sl < slab1; ++sl) {
    const int64_t ts = t_begin + (int64_t)sl * kSlab;
    const bool quant = ts < p.Tq;
    // ---------------- scores of the 16 tokens, as 2 n-tiles of 8
    float acc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
    if (quant) {
      const int64_t grp = ts / p.G;
      if (grp != cur_group) {
        cur_group = grp;
        // folded query of this group: x_c = q_c * s_c, bias = sum_c x_c (q_min - zp_c)
        const uint4* mp = reinterpret_cast<const uint4*>(km + grp * kHeadDim + 32 * j);
        float x[32];
        float amax = 0.0f, bias = 0.0f;
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const uint4 v = __ldg(mp + k);
          const uint32_t ws[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 sz = __half22float2(*reinterpret_cast<const __half2*>(&ws[e]));
            const int c = 4 * k + e;
            x[c] = qf[c] * sz.x;
            bias = fmaf(x[c], qmin - sz.y, bias);
            amax = fmaxf(amax, fabsf(x[c]));
          }
        }
        bias += __shfl_xor_sync(0xffffffffu, bias, 1);
        bias += __shfl_xor_sync(0xffffffffu, bias, 2);
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
        amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
        // power-of-two normalisation: amax * 2^E in [2^14, 2^15)
        int E = 0;
        if (amax > 0.0f) E = 14 - (((__float_as_int(amax) >> 23) & 0xFF) - 127);
        E = max(-100, min(100, E));
        const float up = exp2f((float)E);
        qscale = kTwo24 * exp2f((float)-E) * p.scale_log2;
        qbias = bias * p.scale_log2;
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          split2(x[k_pair_ca<BITS>(2 * ks)] * up, x[k_pair_cb<BITS>(2 * ks)] * up, qa[ks][0], qa[ks][1]);
          split2(x[k_pair_ca<BITS>(2 * ks + 1)] * up, x[k_pair_cb<BITS>(2 * ks + 1)] * up, qa[ks][2], qa[ks][3]);
        }
      }
      uint32_t kw[2][CW];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) load_chunk<BITS>(kc + (ts + 8 * nt + g) * p.rowK + j * (p.rowK / 4), kw[nt]);
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma16816(acc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], k_pair<BITS>(kw[nt], 2 * ks),
                   k_pair<BITS>(kw[nt], 2 * ks + 1));
    } else {
      if (cur_group != -2) {
        cur_group = -2;  // raw query fragments for binary16 residual keys: natural channel pairs
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          qa[ks][0] = h2_bits(__floats2half2_rn(qf[4 * ks + 0], qf[4 * ks + 1]));
          qa[ks][2] = h2_bits(__floats2half2_rn(qf[4 * ks + 2], qf[4 * ks + 3]));
          qa[ks][1] = 0u;
          qa[ks][3] = 0u;
        }
        qscale = p.scale_log2;
        qbias = 0.0f;
      }
      uint32_t kw[2][16];
#pragma unroll
      for (int nt = 0; nt < 2; ++nt) {
        const uint4* rp = reinterpret_cast<const uint4*>(kr + ((ts + 8 * nt + g) % p.R_eff) * kHeadDim + 32 * j);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = __ldg(rp + k);
          kw[nt][4 * k] = v.x; kw[nt][4 * k + 1] = v.y; kw[nt][4 * k + 2] = v.z; kw[nt][4 * k + 3] = v.w;
        }
      }
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int ks = 0; ks < 8; ++ks)
          mma16816(acc[nt], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], kw[nt][2 * ks], kw[nt][2 * ks + 1]);
    }
    // scores (log2 units) of tokens ts + {2j, 2j+1, 8+2j, 9+2j} for query qi
    float s[4];
#pragma unroll
    for (int nt = 0; nt < 2; ++nt)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int64_t t = ts + 8 * nt + 2 * j + e;
        const float v = fmaf(acc[nt][e] + acc[nt][e + 2], qscale, qbias);
        s[2 * nt + e] = (t < t_end) ? v : -__int_as_float(0x7f800000);
      }
    // ---------------- online softmax
    float mx = fmaxf(fmaxf(s[0], s[1]), fmaxf(s[2], s[3]));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float m_new = fmaxf(m_run, mx);
    const bool grew = m_new > m_run;
    if (__any_sync(0xffffffffu, grew)) {
      const float alpha = exp2f(m_run - m_new);  // 0 on the first slab (m_run = -inf)
      l_run *= alpha;
#pragma unroll
      for (int k = 0; k < 4; ++k) beta[k] *= alpha;
      // PV column n belongs to query of row n: alphas of columns 2j, 2j+1 live in rows 2j, 2j+1
      const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * j);
      const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * j + 4);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          o[mt][nt][0] *= a0; o[mt][nt][1] *= a1; o[mt][nt][2] *= a0; o[mt][nt][3] *= a1;
        }
      m_run = m_new;
    }
    float pr[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      pr[k] = exp2f(s[k] - m_run);
      l_run += pr[k];
    }
    // ---------------- values: weights p * s per value group, split into binary16 halves
    uint32_t vw[2][CW];
#pragma unroll
    for (int pr_i = 0; pr_i < 2; ++pr_i)
      load_chunk<BITS>(vc + ((ts >> 1) + 4 * pr_i + j) * 2 * p.rowV + g * (p.rowV / 4), vw[pr_i]);
    uint32_t bf[4][NT][2];
#pragma unroll
    for (int vg = 0; vg < 4; ++vg) {
      if (vg < p.n_vg) {
        float wgt[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int64_t t = ts + (k >> 1) * 8 + 2 * j + (k & 1);
          const float2 sz = __half22float2(vm[t * p.n_vg + vg]);
          wgt[k] = pr[k] * sz.x;
          beta[vg] = fmaf(wgt[k], qmin - sz.y, beta[vg]);
        }
        uint32_t hi0, lo0, hi1, lo1;
        split2(wgt[0], wgt[1], hi0, lo0);
        split2(wgt[2], wgt[3], hi1, lo1);
        if (NT == 1) {
          bf[vg][0][0] = lo_lane ? lo0 : hi0;
          bf[vg][0][1] = lo_lane ? lo1 : hi1;
        } else {
          bf[vg][0][0] = hi0; bf[vg][0][1] = hi1;
          bf[vg][NT - 1][0] = lo0; bf[vg][NT - 1][1] = lo1;
        }
      }
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const int vg = (16 * mt) / p.Gv;
      const uint32_t a0 = v_pair<BITS>(vw[0], 2 * mt), a1 = v_pair<BITS>(vw[0], 2 * mt + 1);
      const uint32_t a2 = v_pair<BITS>(vw[1], 2 * mt), a3 = v_pair<BITS>(vw[1], 2 * mt + 1);
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        uint32_t b0, b1;
        // vg is warp-uniform; select without dynamic register indexing
        b0 = bf[0][nt][0]; b1 = bf[0][nt][1];
        if (vg == 1) { b0 = bf[1][nt][0]; b1 = bf[1][nt][1]; }
        if (vg == 2) { b0 = bf[2][nt][0]; b1 = bf[2][nt][1]; }
        if (vg == 3) { b0 = bf[3][nt][0]; b1 = bf[3][nt][1]; }
        mma16816(o[mt][nt], a0, a1, a2, a3, b0, b1);
      }
    }
  }

  // ---------------- per-warp results -> shared memory
  __shared__ float o_s[kWarps][kMaxGqa][kHeadDim];
  __shared__ float m_s[kWarps][kMaxGqa], l_s[kWarps][kMaxGqa], beta_s[kWarps][kMaxGqa][4];
  __shared__ int last_s;
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
  l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    beta[k] += __shfl_xor_sync(0xffffffffu, beta[k], 1);
    beta[k] += __shfl_xor_sync(0xffffffffu, beta[k], 2);
  }
  if (j == 0 && g < r) {  // row g holds query g for g < r
    m_s[warp][g] = m_run;
    l_s[warp][g] = l_run;
#pragma unroll
    for (int k = 0; k < 4; ++k) beta_s[warp][g][k] = beta[k];
  }
  // PV columns: NT == 1: cols 0..3 hi / 4..7 lo of queries 0..3; NT == 2: tile 0 hi, tile 1 lo of queries 0..7
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    float v[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[e] = o[mt][0][e];
      if (NT == 2) v[e] += o[mt][NT - 1][e];
    }
    if (NT == 1) {
#pragma unroll
      for (int e = 0; e < 4; ++e) v[e] += __shfl_xor_sync(0xffffffffu, v[e], 2);  // lo columns j+2 -> j
    }
    const bool writer = (NT == 2) || (j < 2);
    if (writer) {
      const int i0 = 2 * j, i1 = 2 * j + 1;
      const int c0 = 16 * mt + g, c1 = c0 + 8;
      if (i0 < r) { o_s[warp][i0][c0] = v[0]; o_s[warp][i0][c1] = v[2]; }
      if (i1 < r) { o_s[warp][i1][c0] = v[1]; o_s[warp][i1][c1] = v[3]; }
    }
  }
  __syncthreads();

  // ---------------- CTA merge of the warps; thread = channel (128 threads)
  const int c = threadIdx.x;
  const int vgc = c / p.Gv;
  for (int i = 0; i < r; ++i) {
    float M = -__int_as_float(0x7f800000);
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      if (w * spw < n_slabs) M = fmaxf(M, m_s[w][i]);
    float L = 0.0f, acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      if (w * spw >= n_slabs) continue;  // warp had no tokens
      const float wt = exp2f(m_s[w][i] - M);
      L += wt * l_s[w][i];
      acc += wt * fmaf(o_s[w][i][c], kTwo24, beta_s[w][i][vgc]);
    }
    if (p.n_split == 1) {
      p.out[(qrow0 + i) * kHeadDim + c] = acc / L;
    } else {
      p.ws_o[((qrow0 + i) * p.cap + split) * kHeadDim + c] = acc;
      if (c == 0) p.ws_ml[(qrow0 + i) * p.cap + split] = make_float2(M, L);
    }
  }
  if (p.n_split == 1) return;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const uint32_t ticket = atomicAdd(&p.tickets[slice], 1u);
    last_s = (ticket == (uint32_t)(p.n_split - 1));
  }
  __syncthreads();
  if (!last_s) return;
  __threadfence();
  for (int i = 0; i < r; ++i) {
    const float2* ml = p.ws_ml + (qrow0 + i) * p.cap;
    float M = -__int_as_float(0x7f800000);
    for (int s = 0; s < p.n_split; ++s) M = fmaxf(M, __ldcg(&ml[s]).x);
    float L = 0.0f, acc = 0.0f;
    for (int s = 0; s < p.n_split; ++s) {
      const float2 v = __ldcg(&ml[s]);
      const float wt = exp2f(v.x - M);
      L += wt * v.y;
      acc += wt * __ldcg(&p.ws_o[((qrow0 + i) * p.cap + s) * kHeadDim + c]);
    }
    p.out[(qrow0 + i) * kHeadDim + c] = acc / L;
  }
  if (threadIdx.x == 0) p.tickets[slice] = 0u;
}

template <int BITS>
cudaError_t launch_bits(const DecodeParams& p, cudaStream_t stream) {
  dim3 grid((unsigned)p.n_split, (unsigned)p.H, (unsigned)p.B);
  if (p.r <= 4) decode_mma_kernel<BITS, 1><<<grid, kWarps * 32, 0, stream>>>(p);
  else decode_mma_kernel<BITS, 2><<<grid, kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_mma(const DecodeParams& p, int bits, cudaStream_t stream) {
  switch (bits) {
    case 8: return launch_bits<8>(p, stream);
    case 4: return launch_bits<4>(p, stream);
    default: return launch_bits<2>(p, stream);
  }
}

}  // namespace kvq
