// kvq_quant.cu — quantize / pack / append and dequantize kernels (sm_103a).
//
// The quantizer is the affine scheme of the page "KV Cache Quantization — 8-bit and
// 4-bit", § Integer quantization in one screen, applied per channel over groups of G
// tokens for keys and per token over groups of Gv channels for values ("Sub-8-Bit KV
// Cache Quantization Is Not a Free Lever for an RDNA4 Agent Swarm", § The cache is
// two distributions, not one). Every floating-point step is one explicitly rounded
// binary32 intrinsic (this file is also compiled with -fmad=false), so codes, scales
// and zero points are reproducible bit for bit:
//   s_h = binary16_round_up(max((x_max - x_min) / (q_max - q_min),
//                               max|x| / (2048 - 2^bits)))
//   zp  = q_min - rint(x_min / s_h) -> binary16 (an integer of magnitude <= 2048: exact)
//   u   = clamp(rint(x / s_h) + zp, q_min, q_max) - q_min
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq_common.cuh"
#include "kvq_kernels.h"
#include "kvq_quantizer.cuh"

namespace kvq {
namespace {

using namespace quant;

// Store the 4 codes of channels [4*lane, 4*lane+4) into a key row (natural order).
template <int BITS>
__device__ __forceinline__ void store_k4(uint8_t* row, int lane, const uint32_t* u) {
  if (BITS == 8) {
    reinterpret_cast<uint32_t*>(row)[lane] = u[0] | (u[1] << 8) | (u[2] << 16) | (u[3] << 24);
  } else if (BITS == 4) {
    reinterpret_cast<uint16_t*>(row)[lane] = (uint16_t)(u[0] | (u[1] << 4) | (u[2] << 8) | (u[3] << 12));
  } else {
    row[lane] = (uint8_t)(u[0] | (u[1] << 2) | (u[2] << 4) | (u[3] << 6));
  }
}

// ---------------------------------------------------------------------------
// Keys: one CTA per (group, kv head, batch row); NW warps, warp w holds tokens
// w, w+NW, ... of the group, lane l holds channels [4l, 4l+4). Token rows come from
// the residual window (tokens < s_cur) or from the appended input. 8 warps at 4 CTAs per
// SM in general; 16 warps at 3 CTAs per SM (half the rows per warp: 40 instead of 64
// registers) where a warp has more to do per row (isolated entries: kivi-int4o4 prompt
// append +11 %); without isolated entries the 16-warp CTAs measured slower, with a full
// grid (kivi-int4 -6 %) and at batch 1 (llama8b-int8 -5 %).
// ---------------------------------------------------------------------------
template <int BITS, int G, int NW>
__global__ void __launch_bounds__(32 * NW, NW == 16 ? 3 : 4) k_group_kernel(AppendParams p) {
  constexpr int PER_WARP = G / NW;
  static_assert(PER_WARP % 2 == 0, "rows are split in pairs");
  pdl_wait();
  pdl_allow_dependents();
  const int h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t g = p.group0 + blockIdx.x;
  const int64_t t0 = g * G;
  const int64_t slice = (int64_t)b * p.H + h;

  __shared__ float red_min[NW][kHeadDim];
  __shared__ float red_max[NW][kHeadDim];
  __shared__ float s_sc[kHeadDim];
  __shared__ float s_rs[kHeadDim];
  __shared__ int s_zp[kHeadDim];

  // rows are kept as binary16 pairs (half the registers of binary32): the group
  // min/max of binary16 values is exact in binary16
  uint2 x[PER_WARP];
  __half2 mn2[2], mx2[2];
  // token t < s_cur is a residual row (slot t - A0, where A0 = group0 * G is the start
  // of the flushed window, a multiple of the window), token t >= s_cur input row
  // (b, t - s_cur, h)
  const __half* resid = p.k_resid + (slice * (int64_t)p.R_eff - p.group0 * G) * kHeadDim;
  const __half* in = p.k_in + (((int64_t)b * p.n_new - p.s_cur) * p.H + h) * kHeadDim;
  const int64_t in_stride = (int64_t)p.H * kHeadDim;
#pragma unroll
  for (int k = 0; k < PER_WARP; ++k) {
    const int64_t t = t0 + warp + NW * k;
    const __half* row = (t < p.s_cur) ? resid + t * kHeadDim : in + t * in_stride;
    x[k] = *reinterpret_cast<const uint2*>(row + 4 * lane);
  }
  if (p.kout > 0) {
    // dense-and-sparse keys: every row of the group gives up its kout farthest entries
    // (their binary16 values to the row's entry list after the group metadata) before the
    // per-channel ranges are taken; they become +0 in the dense row
    uint32_t* ent = reinterpret_cast<uint32_t*>(reinterpret_cast<uint8_t*>(p.k_meta) + slice * p.k_meta_slice +
                                                (p.S_pad / G) * kHeadDim * 4);
#pragma unroll
    for (int k = 0; k < PER_WARP; k += 2) {  // rows in pairs: one sort of their packed order keys
      const int64_t t = t0 + warp + NW * k;     // row k + 1 is token t + NW
      const uint32_t xa[4] = {x[k].x & 0xFFFFu, x[k].x >> 16, x[k].y & 0xFFFFu, x[k].y >> 16};
      const uint32_t xc[4] = {x[k + 1].x & 0xFFFFu, x[k + 1].x >> 16, x[k + 1].y & 0xFFFFu, x[k + 1].y >> 16};
      bool ta[4], tc[4];
      split_two_rows_outliers(xa, xc, ta, tc, ent + t * p.kout, ent + (t + NW) * p.kout, p.kout, lane);
      x[k].x &= (ta[0] ? 0xFFFF0000u : 0xFFFFFFFFu) & (ta[1] ? 0x0000FFFFu : 0xFFFFFFFFu);
      x[k].y &= (ta[2] ? 0xFFFF0000u : 0xFFFFFFFFu) & (ta[3] ? 0x0000FFFFu : 0xFFFFFFFFu);
      x[k + 1].x &= (tc[0] ? 0xFFFF0000u : 0xFFFFFFFFu) & (tc[1] ? 0x0000FFFFu : 0xFFFFFFFFu);
      x[k + 1].y &= (tc[2] ? 0xFFFF0000u : 0xFFFFFFFFu) & (tc[3] ? 0x0000FFFFu : 0xFFFFFFFFu);
    }
  }
#pragma unroll
  for (int k = 0; k < PER_WARP; ++k) {
    const __half2 a = *reinterpret_cast<const __half2*>(&x[k].x), c = *reinterpret_cast<const __half2*>(&x[k].y);
    if (k == 0) {
      mn2[0] = a; mx2[0] = a; mn2[1] = c; mx2[1] = c;
    } else {
      mn2[0] = __hmin2(mn2[0], a); mx2[0] = __hmax2(mx2[0], a);
      mn2[1] = __hmin2(mn2[1], c); mx2[1] = __hmax2(mx2[1], c);
    }
  }
  float mn[4], mx[4];
  mn[0] = __low2float(mn2[0]); mn[1] = __high2float(mn2[0]); mn[2] = __low2float(mn2[1]); mn[3] = __high2float(mn2[1]);
  mx[0] = __low2float(mx2[0]); mx[1] = __high2float(mx2[0]); mx[2] = __low2float(mx2[1]); mx[3] = __high2float(mx2[1]);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    red_min[warp][4 * lane + e] = mn[e];
    red_max[warp][4 * lane + e] = mx[e];
  }
  __syncthreads();
  if (threadIdx.x < kHeadDim) {
    const int c = threadIdx.x;
    float a = red_min[0][c], z = red_max[0][c];
#pragma unroll
    for (int w = 1; w < NW; ++w) {
      a = fminf(a, red_min[w][c]);
      z = fmaxf(z, red_max[w][c]);
    }
    __half s_h, z_h;
    float s, rs, zp;
    group_params<BITS>(a, z, s_h, z_h, s, rs, zp);
    s_sc[c] = s;
    s_rs[c] = rs;
    s_zp[c] = (int)zp - (int)Q<BITS>::qmin;
    reinterpret_cast<__half2*>(reinterpret_cast<uint8_t*>(p.k_meta) + slice * p.k_meta_slice)[g * kHeadDim + c] =
        __halves2half2(s_h, z_h);
  }
  __syncthreads();
  float s[4], rs[4];
  int zp[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    s[e] = s_sc[4 * lane + e];
    rs[e] = s_rs[4 * lane + e];
    zp[e] = s_zp[4 * lane + e];
  }
  uint8_t* codes = p.k_codes + slice * p.k_codes_slice;
#pragma unroll
  for (int k = 0; k < PER_WARP; ++k) {
    const int64_t t = t0 + warp + NW * k;
    float xf[4];
    load4(reinterpret_cast<const __half*>(&x[k]), xf);
    uint32_t u[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) u[e] = quant_code<BITS>(xf[e], s[e], rs[e], zp[e]);
    store_k4<BITS>(codes + t * (kHeadDim * BITS / 8), lane, u);
  }
}

// ---------------------------------------------------------------------------
// Keys in groups of 32 tokens: one warp per (group, kv head, batch row), eight groups of
// one (kv head, batch row) per CTA. Lane l holds channels [4l, 4l+4) of all 32 rows of
// its group as binary16 pairs, so each channel's min and max are taken inside the lane
// (exact in binary16) and the lane computes its four channels' parameters itself: no
// shared memory, no CTA barrier. Rows as in k_group_kernel; without isolated key entries
// (with them, k_group_kernel<BITS, 32> splits the rows first).
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(256, 2) k_group32_kernel(AppendParams p) {
  constexpr int G = 32;
  pdl_wait();
  pdl_allow_dependents();
  const int h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = (int)blockIdx.x * 8 + warp;
  if (gi >= p.n_groups) return;  // whole warp
  const int64_t g = p.group0 + gi;
  const int64_t t0 = g * G;
  const int64_t slice = (int64_t)b * p.H + h;

  uint2 x[G];  // row k = token t0 + k, channels [4 lane, 4 lane + 4)
  const __half* resid = p.k_resid + (slice * (int64_t)p.R_eff - p.group0 * G) * kHeadDim;
  const __half* in = p.k_in + (((int64_t)b * p.n_new - p.s_cur) * p.H + h) * kHeadDim;
  const int64_t in_stride = (int64_t)p.H * kHeadDim;
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const int64_t t = t0 + k;
    const __half* row = (t < p.s_cur) ? resid + t * kHeadDim : in + t * in_stride;
    x[k] = *reinterpret_cast<const uint2*>(row + 4 * lane);
  }
  __half2 mn2[2], mx2[2];
#pragma unroll
  for (int k = 0; k < G; ++k) {
    const __half2 a = *reinterpret_cast<const __half2*>(&x[k].x), c = *reinterpret_cast<const __half2*>(&x[k].y);
    mn2[0] = k ? __hmin2(mn2[0], a) : a;
    mx2[0] = k ? __hmax2(mx2[0], a) : a;
    mn2[1] = k ? __hmin2(mn2[1], c) : c;
    mx2[1] = k ? __hmax2(mx2[1], c) : c;
  }
  const float mn[4] = {__low2float(mn2[0]), __high2float(mn2[0]), __low2float(mn2[1]), __high2float(mn2[1])};
  const float mx[4] = {__low2float(mx2[0]), __high2float(mx2[0]), __low2float(mx2[1]), __high2float(mx2[1])};
  float s[4], rs[4];
  int zp[4];
  uint32_t meta[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    __half s_h, z_h;
    float zpf;
    group_params<BITS>(mn[e], mx[e], s_h, z_h, s[e], rs[e], zpf);
    zp[e] = (int)zpf - (int)Q<BITS>::qmin;
    meta[e] = (uint32_t)__half_as_ushort(s_h) | ((uint32_t)__half_as_ushort(z_h) << 16);
  }
  // (scale, zero point) of channels [4 lane, 4 lane + 4): 16 bytes
  *reinterpret_cast<uint4*>(reinterpret_cast<uint8_t*>(p.k_meta) + slice * p.k_meta_slice +
                            (g * kHeadDim + 4 * lane) * 4) = make_uint4(meta[0], meta[1], meta[2], meta[3]);
  uint8_t* codes = p.k_codes + slice * p.k_codes_slice;
#pragma unroll
  for (int k = 0; k < G; ++k) {
    float xf[4];
    load4(reinterpret_cast<const __half*>(&x[k]), xf);
    uint32_t u[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) u[e] = quant_code<BITS>(xf[e], s[e], rs[e], zp[e]);
    store_k4<BITS>(codes + (t0 + k) * (kHeadDim * BITS / 8), lane, u);
  }
}

// ---------------------------------------------------------------------------
// Values (and the key residual copy): each warp quantizes four appended (batch row,
// token, kv head) rows, in the input's own order; lanes 8r .. 8r+7 hold row r, lane
// 8r + l its channels [16l, 16l + 16). A value group of Gv channels spans Gv/16 lanes.
// In the pair-row layout channel 16l + i sits at position 16(i % 8) + 2l + i / 8, so
// 8-bit codes fill their 16-bit units within a lane and 4-bit units take two lanes (2-bit
// values: v_token32_kernel). SYM: the symmetric per-token scheme (one group of d channels,
// scale from max|x|, zero point 0).
// ---------------------------------------------------------------------------
template <int BITS, bool SYM = false, int LPG = 8>
__global__ void __launch_bounds__(256, 8) v_token_kernel(AppendParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sl = lane & 7;
  // rows of batch row b = blockIdx.y in the input's order (token, kv head)
  const int64_t nb = p.n_new * p.H;
  const int64_t wb_raw = ((int64_t)blockIdx.x * 8 + warp) * 4 + (lane >> 3);
  pdl_wait();
  pdl_allow_dependents();
  const bool valid = wb_raw < nb;
  const int64_t wb = valid ? wb_raw : nb - 1;  // lanes past the end read a real row and store nothing
  int64_t tt;
  int h;
  if (p.rows_32) {
    tt = fast_div((uint32_t)wb, p.fd_H);
    h = (int)(wb - tt * p.H);
  } else {
    tt = wb / p.H;
    h = (int)(wb % p.H);
  }
  const int b = blockIdx.y;
  const int64_t w = (int64_t)b * nb + wb;
  const int64_t t = p.s_cur + tt;
  const int64_t slice = (int64_t)b * p.H + h;

  uint32_t wd[8];    // channels 16 sl + 2k, 16 sl + 2k + 1 as a binary16 pair
  __half2 mn2, mx2;  // the lane's min and max in binary16 (exact), per half of the pairs
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.v_in + w * kHeadDim + 16 * sl);
    const uint4 a = src[0], c = src[1];
    wd[0] = a.x; wd[1] = a.y; wd[2] = a.z; wd[3] = a.w; wd[4] = c.x; wd[5] = c.y; wd[6] = c.z; wd[7] = c.w;
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const __half2 hk = *reinterpret_cast<const __half2*>(&wd[k]);
      mn2 = k ? __hmin2(mn2, hk) : hk;
      mx2 = k ? __hmax2(mx2, hk) : hk;
    }
  }
  constexpr int lpg = LPG;  // lanes per value group (Gv / 16): 2, 4 or 8
  __half s_h, z_h;
  float s, rs, zp;
  if constexpr (SYM) {
    const __half2 am = __hmax2(__habs2(mn2), __habs2(mx2));
    float a = fmaxf(__low2float(am), __high2float(am));
#pragma unroll
    for (int off = 1; off < 8; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    sym_params8(a, s_h, s, rs);
    z_h = __float2half_rn(0.0f);
    zp = 0.0f;
  } else {
    float mn = fminf(__low2float(mn2), __high2float(mn2)), mx = fmaxf(__low2float(mx2), __high2float(mx2));
#pragma unroll
    for (int off = 1; off < lpg; off <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    group_params<BITS>(mn, mx, s_h, z_h, s, rs, zp);
  }
  if (valid && sl % lpg == 0) {  // the token's half of its pair's record for this group
    __half* rec = reinterpret_cast<__half*>(p.v_meta) + ((slice * (p.S_pad >> 1) + (t >> 1)) * p.n_vg + sl / lpg) * 4 +
                  (int)(t & 1);
    rec[0] = s_h;
    rec[2] = z_h;
  }
  const int zpu = (int)zp - (int)Q<BITS>::qmin;
  uint32_t u[16];
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wd[k]));
    u[2 * k] = quant_code<BITS>(f.x, s, rs, zpu);
    u[2 * k + 1] = quant_code<BITS>(f.y, s, rs, zpu);
  }

  uint16_t* pair =
      reinterpret_cast<uint16_t*>(p.v_codes + slice * p.v_codes_slice + (t >> 1) * (2 * kHeadDim * BITS / 8)) + (t & 1);
  static_assert(BITS == 8 || BITS == 4, "2-bit values: v_token32_kernel");
  if (BITS == 8) {
    // unit 8m + l = (channel 16l + m, channel 16l + m + 8)
    if (valid) {
#pragma unroll
      for (int m = 0; m < 8; ++m) pair[2 * (8 * m + sl)] = (uint16_t)(u[m] | (u[m + 8] << 8));
    }
  } else if (BITS == 4) {
    // unit 4m + l/2: bytes of lanes 2(l/2) (low) and 2(l/2) + 1 (high); byte m of a lane
    // holds channels 16l + m and 16l + m + 8. Even lanes store m = 0..3, odd lanes 4..7.
    uint32_t w0 = 0, w1 = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      w0 |= (u[m] | (u[m + 8] << 4)) << (8 * m);
      w1 |= (u[m + 4] | (u[m + 12] << 4)) << (8 * m);
    }
    const bool odd = sl & 1;
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? w0 : w1, 1);
    const uint32_t lo = odd ? recv : w0, hi = odd ? w1 : recv;
    if (valid) {
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int m = odd ? 4 + j : j;
        pair[2 * (4 * m + (sl >> 1))] = (uint16_t)__byte_perm(lo, hi, (unsigned)(j | ((4 + j) << 4)));
      }
    }
  }
  // Keys of tokens past the last full residual window go to the residual.
  if (!SYM && valid && t >= p.A1) {
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_in + w * kHeadDim + 16 * sl);
    uint4* kd = reinterpret_cast<uint4*>(p.k_resid + (slice * p.R_eff + (t - p.A1)) * kHeadDim + 16 * sl);
    kd[0] = ks[0];
    kd[1] = ks[1];
  }
}

// ---------------------------------------------------------------------------
// 2-bit values (and the key residual copy): each warp quantizes eight appended (batch
// row, token, kv head) rows, in the input's own order; lanes 4r .. 4r+3 hold row r, lane
// 4r + l its channels [32l, 32l + 32) as binary16 pairs (converted to binary32 one pair at
// a time where they are quantized). A value group of Gv channels spans Gv/32 lanes. In the
// pair-row layout channel 32l + 8q + m (m < 8, q < 4) sits at position 16m + 4l + q, so a
// lane's four codes of one m fill one byte of a 16-bit unit whose other byte is lane
// l ^ 1's. Twice the channels per lane of v_token_kernel halve the per-row work per code
// (the group parameters, the row index), which pays for 2-bit codes; with 4-bit codes
// (each lane then fills whole units) it measured 6 % slower than v_token_kernel.
// ---------------------------------------------------------------------------
template <int BITS>
__global__ void __launch_bounds__(256, 6) v_token32_kernel(AppendParams p) {
  static_assert(BITS == 2, "2-bit codes only");
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sl = lane & 3;
  // rows of batch row b = blockIdx.y in the input's order (token, kv head)
  const int64_t nb = p.n_new * p.H;
  const int64_t wb_raw = ((int64_t)blockIdx.x * 8 + warp) * 8 + (lane >> 2);
  pdl_wait();
  pdl_allow_dependents();
  const bool valid = wb_raw < nb;
  const int64_t wb = valid ? wb_raw : nb - 1;  // lanes past the end read a real row and store nothing
  int64_t tt;
  int h;
  if (p.rows_32) {
    tt = fast_div((uint32_t)wb, p.fd_H);
    h = (int)(wb - tt * p.H);
  } else {
    tt = wb / p.H;
    h = (int)(wb % p.H);
  }
  const int b = blockIdx.y;
  const int64_t w = (int64_t)b * nb + wb;
  const int64_t t = p.s_cur + tt;
  const int64_t slice = (int64_t)b * p.H + h;

  uint32_t xh[16];   // channels 32 sl + 2k and 32 sl + 2k + 1 as a binary16 pair
  __half2 mn2, mx2;  // the lane's min and max in binary16 (exact), per half of the pairs
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.v_in + w * kHeadDim + 32 * sl);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) {
      const uint4 a = src[k4];
      xh[4 * k4] = a.x; xh[4 * k4 + 1] = a.y; xh[4 * k4 + 2] = a.z; xh[4 * k4 + 3] = a.w;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const __half2 hk = *reinterpret_cast<const __half2*>(&xh[4 * k4 + k]);
        mn2 = (k4 | k) ? __hmin2(mn2, hk) : hk;
        mx2 = (k4 | k) ? __hmax2(mx2, hk) : hk;
      }
    }
  }
  const float mn0 = fminf(__low2float(mn2), __high2float(mn2)), mx0 = fmaxf(__low2float(mx2), __high2float(mx2));
  const int lpg = p.Gv >> 5;  // lanes per value group: 1, 2 or 4
  __half s_h, z_h;
  float s, rs, zp;
  {
    float mn = mn0, mx = mx0;
    for (int off = 1; off < lpg; off <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    group_params<BITS>(mn, mx, s_h, z_h, s, rs, zp);
  }
  if (valid && sl % lpg == 0) {  // the token's half of its pair's record for this group
    __half* rec = reinterpret_cast<__half*>(p.v_meta) + ((slice * (p.S_pad >> 1) + (t >> 1)) * p.n_vg + sl / lpg) * 4 +
                  (int)(t & 1);
    rec[0] = s_h;
    rec[2] = z_h;
  }
  const int zpu = (int)zp - (int)Q<BITS>::qmin;
  // codes of channels 32 sl + 8q + m and + 1 (m even), from one binary16 pair
  auto codes2 = [&](int q, int m, uint32_t& c0, uint32_t& c1) {
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&xh[(8 * q + m) >> 1]));
    c0 = quant_code<BITS>(f.x, s, rs, zpu);
    c1 = quant_code<BITS>(f.y, s, rs, zpu);
  };

  // the token's half of its pair row: 16-bit unit k at pair[2 k]
  uint16_t* pair =
      reinterpret_cast<uint16_t*>(p.v_codes + slice * p.v_codes_slice + (t >> 1) * (2 * kHeadDim * BITS / 8)) + (t & 1);
  {
    // unit 2m + sl/2: this lane's codes q = 0..3 at bits 2q of byte (sl & 1). Bytes of
    // m = 0..3 and 4..7 are gathered in two words; even lanes store m = 0..3, odd lanes
    // m = 4..7, each taking the other byte of its units from lane sl ^ 1.
    uint32_t wm[2] = {0u, 0u};
#pragma unroll
    for (int m = 0; m < 8; m += 2) {
      uint32_t b0 = 0, b1 = 0;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint32_t c0, c1;
        codes2(q, m, c0, c1);
        b0 |= c0 << (2 * q);
        b1 |= c1 << (2 * q);
      }
      wm[m >> 2] |= (b0 | (b1 << 8)) << (8 * (m & 3));
    }
    const bool odd = sl & 1;
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, odd ? wm[0] : wm[1], 1);
    const uint32_t lo = odd ? recv : wm[0], hi = odd ? wm[1] : recv;  // even lane's bytes, odd lane's bytes
    if (valid) {
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        const int m = (odd ? 4 : 0) + jj;
        pair[2 * (2 * m + (sl >> 1))] = (uint16_t)__byte_perm(lo, hi, (unsigned)(jj | ((4 + jj) << 4)));
      }
    }
  }
  // Keys of tokens past the last full residual window go to the residual.
  if (valid && t >= p.A1) {
    const uint4* ks = reinterpret_cast<const uint4*>(p.k_in + w * kHeadDim + 32 * sl);
    uint4* kd = reinterpret_cast<uint4*>(p.k_resid + (slice * p.R_eff + (t - p.A1)) * kHeadDim + 32 * sl);
#pragma unroll
    for (int k4 = 0; k4 < 4; ++k4) kd[k4] = ks[k4];
  }
}

// ---------------------------------------------------------------------------
// Symmetric per-token keys ("KV Cache Quantization — 8-bit and 4-bit", § Symmetric vs
// asymmetric; one scale per token, "Sub-8-Bit KV Cache Quantization Is Not a Free Lever
// for an RDNA4 Agent Swarm", § The RDNA4 kernel angle): four appended rows per warp in
// the input's order, lane 8r + l holding channels [16l, 16l + 16) of row r; the 8-bit
// codes go to the key row in channel order (16 bytes per lane), the binary16 scale to
// k_meta[slice][t].
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_token_sym_kernel(AppendParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int sl = lane & 7;
  const int64_t nb = p.n_new * p.H;
  const int64_t wb_raw = ((int64_t)blockIdx.x * 8 + warp) * 4 + (lane >> 3);
  pdl_wait();
  pdl_allow_dependents();
  const bool valid = wb_raw < nb;
  const int64_t wb = valid ? wb_raw : nb - 1;  // lanes past the end read a real row and store nothing
  int64_t tt;
  int h;
  if (p.rows_32) {  // a 64-bit division costs a call to a long software routine
    tt = fast_div((uint32_t)wb, p.fd_H);
    h = (int)(wb - tt * p.H);
  } else {
    tt = wb / p.H;
    h = (int)(wb % p.H);
  }
  const int b = blockIdx.y;
  const int64_t w = (int64_t)b * nb + wb;
  const int64_t t = p.s_cur + tt;
  const int64_t slice = (int64_t)b * p.H + h;
  float x[16];
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.k_in + w * kHeadDim + 16 * sl);
    const uint4 a = src[0], c = src[1];
    const uint32_t wd[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&wd[k]));
      x[2 * k] = f.x;
      x[2 * k + 1] = f.y;
    }
  }
  float a = fabsf(x[0]);
#pragma unroll
  for (int i = 1; i < 16; ++i) a = fmaxf(a, fabsf(x[i]));
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  __half s_h;
  float s, rs;
  sym_params8(a, s_h, s, rs);
  uint32_t wv[4] = {0u, 0u, 0u, 0u};
#pragma unroll
  for (int i = 0; i < 16; ++i) wv[i >> 2] |= quant_code<8>(x[i], s, rs, 128) << (8 * (i & 3));
  if (valid) {
    *reinterpret_cast<uint4*>(p.k_codes + slice * p.k_codes_slice + t * p.rowK + 16 * sl) =
        make_uint4(wv[0], wv[1], wv[2], wv[3]);
    if (sl == 0) reinterpret_cast<__half*>(reinterpret_cast<uint8_t*>(p.k_meta) + slice * p.k_meta_slice)[t] = s_h;
  }
}

// ---------------------------------------------------------------------------
// Symmetric per-token keys with outlier isolation (kout > 0): two rows per warp (the
// median and the farthest entries need the whole row; the two rows' medians come from one
// sort of their packed order keys), see quant::split_two_rows_outliers.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) k_token_sym_outlier_kernel(AppendParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t nb = p.n_new * p.H;
  const int64_t wb0 = ((int64_t)blockIdx.x * 8 + warp) * 2;
  pdl_wait();
  pdl_allow_dependents();
  if (wb0 >= nb) return;  // whole warp
  const int b = blockIdx.y;
  const int n_rows = wb0 + 1 < nb ? 2 : 1;
  uint32_t xb[2][4];
  float x[2][4];
  uint8_t* codes[2];
  uint8_t* kmb[2];
  int64_t t[2];
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int64_t wb = k < n_rows ? wb0 + k : wb0;  // a lone last row is split twice, stored once
    int64_t tt;
    int h;
    if (p.rows_32) {
      tt = fast_div((uint32_t)wb, p.fd_H);
      h = (int)(wb - tt * p.H);
    } else {
      tt = wb / p.H;
      h = (int)(wb % p.H);
    }
    const int64_t slice = (int64_t)b * p.H + h;
    t[k] = p.s_cur + tt;
    codes[k] = p.k_codes + slice * p.k_codes_slice + t[k] * p.rowK;
    kmb[k] = reinterpret_cast<uint8_t*>(p.k_meta) + slice * p.k_meta_slice;
    const __half* row = p.k_in + ((int64_t)b * nb + wb) * kHeadDim + 4 * lane;
    const uint2 raw = *reinterpret_cast<const uint2*>(row);
    xb[k][0] = raw.x & 0xFFFFu; xb[k][1] = raw.x >> 16; xb[k][2] = raw.y & 0xFFFFu; xb[k][3] = raw.y >> 16;
    load4(row, x[k]);
  }
  bool taken[2][4];
  uint32_t* ent0 = reinterpret_cast<uint32_t*>(kmb[0] + p.S_pad * 2) + t[0] * p.kout;
  uint32_t* ent1 = reinterpret_cast<uint32_t*>(kmb[1] + p.S_pad * 2) + t[1] * p.kout;
  split_two_rows_outliers(xb[0], xb[1], taken[0], taken[1], ent0, ent1, p.kout, lane);
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    if (k >= n_rows) break;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (taken[k][e]) x[k][e] = 0.0f;
    quantize_sym_row(x[k], codes[k], reinterpret_cast<__half*>(kmb[k]) + t[k], lane);
  }
}

// ---------------------------------------------------------------------------
// Dequantize the first T tokens: one warp per (batch row, kv head, token).
// x_hat = s * (u + q_min - zp), one binary32 product.
// ---------------------------------------------------------------------------
template <int BITS, int VBITS>
__global__ void __launch_bounds__(256) dequant_kernel(DequantParams p, int64_t n_rows) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t w = (int64_t)blockIdx.x * 8 + warp;
  if (w >= n_rows) return;
  const int64_t t = w % p.T;
  const int64_t slice = w / p.T;  // b * H + h
  const int c0 = 4 * lane;
  float kx[4], vx[4];
  if (p.sym) {  // symmetric per-token keys: x_hat = s_t * (u + q_min)
    const uint8_t* row = p.k_codes + slice * p.k_codes_slice + t * p.rowK;
    const uint8_t* kmb = reinterpret_cast<const uint8_t*>(p.k_meta) + slice * p.k_meta_slice;
    const float s = __half2float(reinterpret_cast<const __half*>(kmb)[t]);
#pragma unroll
    for (int e = 0; e < 4; ++e) kx[e] = __fmul_rn(s, (float)((int)row[c0 + e] - 128));
    // isolated entries: the stored binary16 value (the dense x_hat there is 0)
    const uint32_t* ent = reinterpret_cast<const uint32_t*>(kmb + p.S_pad * 2) + t * p.kout;
    for (int r = 0; r < p.kout; ++r) {
      const uint32_t en = ent[r];
      const int c = (int)(en & 0xFFFFu);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (c == c0 + e) kx[e] = __fadd_rn(kx[e], __half2float(__ushort_as_half((unsigned short)(en >> 16))));
    }
  } else if (t < p.Tq) {
    const uint8_t* row = p.k_codes + slice * p.k_codes_slice + t * p.rowK;
    const __half2* meta = reinterpret_cast<const __half2*>(reinterpret_cast<const uint8_t*>(p.k_meta) +
                                                           slice * p.k_meta_slice) + (t / p.G) * kHeadDim;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = c0 + e;
      const uint32_t u = (row[(c * BITS) >> 3] >> ((c * BITS) & 7)) & ((1u << BITS) - 1u);
      const __half2 m = meta[c];
      kx[e] = __fmul_rn(__low2float(m), __fsub_rn((float)((int)u + (int)Q<BITS>::qmin), __high2float(m)));
    }
    // isolated entries after the group metadata: the stored binary16 value is added to the
    // dense x_hat there (the dense row held +0 at that channel)
    const uint32_t* ent = reinterpret_cast<const uint32_t*>(reinterpret_cast<const uint8_t*>(p.k_meta) +
                                                            slice * p.k_meta_slice + (p.S_pad / p.G) * kHeadDim * 4) +
                          t * p.kout;
    for (int r = 0; r < p.kout; ++r) {
      const uint32_t en = ent[r];
      const int c = (int)(en & 0xFFFFu);
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (c == c0 + e) kx[e] = __fadd_rn(kx[e], __half2float(__ushort_as_half((unsigned short)(en >> 16))));
    }
  } else {
    load4(p.k_resid + (slice * p.R_eff + t % p.R_eff) * kHeadDim + c0, kx);
  }
  {
    const uint16_t* pair = reinterpret_cast<const uint16_t*>(p.v_codes + slice * p.v_codes_slice + (t >> 1) * 2 * p.rowV);
    // the pair's records {scale 2p, scale 2p+1, zp 2p, zp 2p+1}, one per group
    const __half* rec = reinterpret_cast<const __half*>(p.v_meta) + (slice * (p.S_pad >> 1) + (t >> 1)) * p.n_vg * 4 +
                        (int)(t & 1);
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int c = c0 + e;
      const int pos = 16 * (c & 7) + 2 * (c >> 4) + ((c >> 3) & 1);
      const int bit = pos * VBITS;
      const uint32_t unit = pair[2 * (bit >> 4) + (int)(t & 1)];
      const uint32_t u = (unit >> (bit & 15)) & ((1u << VBITS) - 1u);
      const int jg = c / p.Gv;
      vx[e] = __fmul_rn(__half2float(rec[4 * jg]),
                        __fsub_rn((float)((int)u + (int)Q<VBITS>::qmin), __half2float(rec[4 * jg + 2])));
    }
  }
  *reinterpret_cast<float4*>(p.k_out + w * kHeadDim + c0) = make_float4(kx[0], kx[1], kx[2], kx[3]);
  *reinterpret_cast<float4*>(p.v_out + w * kHeadDim + c0) = make_float4(vx[0], vx[1], vx[2], vx[3]);
}

template <int BITS>
cudaError_t launch_keys(const AppendParams& p, cudaStream_t stream) {
  if (p.n_groups <= 0) return cudaSuccess;
  dim3 grid((unsigned)p.n_groups, (unsigned)p.H, (unsigned)p.B);
  switch (p.G) {
    case 32:
      if (p.kout > 0) return launch_pdl(k_group_kernel<BITS, 32, 16>, grid, dim3(512), 0, stream, p);
      return launch_pdl(k_group32_kernel<BITS>, dim3((unsigned)((p.n_groups + 7) / 8), (unsigned)p.H, (unsigned)p.B),
                        dim3(256), 0, stream, p);
    case 64:
      return p.wide_keys ? launch_pdl(k_group_kernel<BITS, 64, 16>, grid, dim3(512), 0, stream, p)
                         : launch_pdl(k_group_kernel<BITS, 64, 8>, grid, dim3(256), 0, stream, p);
    default:
      return p.wide_keys ? launch_pdl(k_group_kernel<BITS, 128, 16>, grid, dim3(512), 0, stream, p)
                         : launch_pdl(k_group_kernel<BITS, 128, 8>, grid, dim3(256), 0, stream, p);
  }
}

template <int VBITS, bool SYM = false>
cudaError_t launch_values(const AppendParams& p, cudaStream_t stream) {
  const int64_t rows = p.n_new * p.H;  // per batch row
  if constexpr (VBITS == 2 && !SYM) {
    return launch_pdl(v_token32_kernel<VBITS>, dim3((unsigned)((rows + 63) / 64), (unsigned)p.B), dim3(256), 0, stream,
                      p);
  } else {
    const dim3 grid((unsigned)((rows + 31) / 32), (unsigned)p.B);
    if constexpr (SYM) return launch_pdl(v_token_kernel<VBITS, true, 8>, grid, dim3(256), 0, stream, p);
    switch (p.Gv) {  // lanes per value group as a constant: the group reduction unrolls
      case 32: return launch_pdl(v_token_kernel<VBITS, false, 2>, grid, dim3(256), 0, stream, p);
      case 64: return launch_pdl(v_token_kernel<VBITS, false, 4>, grid, dim3(256), 0, stream, p);
      default: return launch_pdl(v_token_kernel<VBITS, false, 8>, grid, dim3(256), 0, stream, p);
    }
  }
}

template <int BITS, int VBITS>
cudaError_t launch_dequant_bits(const DequantParams& p, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.B * p.H * p.T;
  dequant_kernel<BITS, VBITS><<<(unsigned)((rows + 7) / 8), 256, 0, stream>>>(p, rows);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_append(const AppendParams& p, int bits, int vbits, cudaStream_t stream) {
  if (p.sym) {  // symmetric per-token int8: keys and values quantized per token
    const int64_t rows = p.n_new * p.H;
    cudaError_t e = p.kout > 0 ? launch_pdl(k_token_sym_outlier_kernel, dim3((unsigned)((rows + 15) / 16), (unsigned)p.B),
                                            dim3(256), 0, stream, p)
                               : launch_pdl(k_token_sym_kernel, dim3((unsigned)((rows + 31) / 32), (unsigned)p.B),
                                            dim3(256), 0, stream, p);
    if (e != cudaSuccess) return e;
    e = launch_values<8, true>(p, stream);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
  }
  cudaError_t e = bits == 8 ? launch_keys<8>(p, stream) : (bits == 4 ? launch_keys<4>(p, stream) : launch_keys<2>(p, stream));
  if (e != cudaSuccess) return e;
  e = vbits == 8 ? launch_values<8>(p, stream) : (vbits == 4 ? launch_values<4>(p, stream) : launch_values<2>(p, stream));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_dequant(const DequantParams& p, int bits, int vbits, cudaStream_t stream) {
  if (vbits != bits) return launch_dequant_bits<8, 4>(p, stream);  // the one mixed configuration
  switch (bits) {
    case 8: return launch_dequant_bits<8, 8>(p, stream);
    case 4: return launch_dequant_bits<4, 4>(p, stream);
    default: return launch_dequant_bits<2, 2>(p, stream);
  }
}

}  // namespace kvq
