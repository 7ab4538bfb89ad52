// kvq_quantizer.cuh — the bit-exact affine quantizer shared by the append kernels and
// the fused decode step (library-internal).
//
// The quantizer is the affine scheme of the page "KV Cache Quantization — 8-bit and
// 4-bit", § Integer quantization in one screen. Every floating-point step is one
// explicitly rounded binary32 intrinsic, so no compiler contraction can change a
// result and codes, scales and zero points are reproducible bit for bit:
//   s_h = binary16_round_up(max((x_max - x_min) / (q_max - q_min),
//                               max|x| / (2048 - 2^bits)))
//   zp  = q_min - rint(x_min / s_h) -> binary16 (an integer of magnitude <= 2048: exact)
//   u   = clamp(rint(x / s_h) + zp, q_min, q_max) - q_min
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kvq_common.cuh"

namespace kvq {
namespace quant {

template <int BITS>
struct Q {
  static constexpr float qmin = -(float)(1 << (BITS - 1));
  static constexpr float qmax = (float)((1 << (BITS - 1)) - 1);
};

// Correctly rounded binary32 quotient a / b from the correctly rounded reciprocal
// rb = RN(1/b), by Markstein's fma correction (P. W. Markstein, "Computation of
// elementary functions on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1),
// 1990): q0 = RN(a * rb) lies within 1.5 ulp of a/b, the remainder a - b*q0 is exactly
// representable (one fma computes it), and q0 + remainder*rb = a/b + e with
// |e| <= 1.5 * 2^-24 ulp, so the final fma returns RN(a/b) whenever a/b, if it is not a
// binary32 number, lies farther than that from every rounding midpoint (a = -0 gives
// +0; every use rounds the quotient to an integer and adds one, so the sign of a zero
// quotient never shows). The two uses:
//  * a and b binary16 values (11-bit significands; the quantizer's x/s and x_min/s):
//    the remainder is a multiple of ulp(b)*ulp(q0) below 2^12 of them, and such a
//    quotient lies at least 2^-12 ulp from every midpoint;
//  * a any positive binary32 and b = 2^bits - 1 (odd, at most 8 bits; the scale's
//    range/levels): the remainder is an integer multiple of ulp(a/b) below 2^9 of them,
//    and a - m*b is an odd multiple of ulp(a/b)/2 for every midpoint m, so the quotient
//    lies at least 2^-9 ulp from every midpoint;
//  * a a positive binary16 value and b = 2048 - 2^bits (the far-group scale floor): b is
//    a power of two times an odd number of at most 9 bits, and a quotient that is not a
//    binary32 number lies at least 2^-10 ulp from every midpoint.
__device__ __forceinline__ float div_rn(float a, float b, float rb) {
  const float q0 = __fmul_rn(a, rb);
  const float r = __fmaf_rn(-b, q0, a);
  return __fmaf_rn(r, rb, q0);
}

// RN(1 / (2^BITS - 1)) as binary32 bit patterns.
template <int BITS>
__device__ __forceinline__ float inv_levels() {
  return __int_as_float(BITS == 8 ? 0x3B808081 : (BITS == 4 ? 0x3D888889 : 0x3EAAAAAB));
}
// RN(1 / (2048 - 2^BITS)) as binary32 bit patterns.
template <int BITS>
__device__ __forceinline__ float inv_far() {
  return __int_as_float(BITS == 8 ? 0x3A124925 : (BITS == 4 ? 0x3A010204 : 0x3A004020));
}

// Group parameters from the (exact) binary32 min and max of binary16 inputs:
// binary16 scale s_h and zero point z_h, and as binary32 s, rs = RN(1/s), zp.
template <int BITS>
__device__ __forceinline__ void group_params(float xmin, float xmax, __half& s_h, __half& z_h, float& s, float& rs,
                                             float& zp) {
  // a constant group is widened to include 0 (selects, not branches: every lane takes the
  // same instructions; fminf/fmaxf may differ from the comparisons only in the sign of a
  // zero, which changes neither the range nor the zero point)
  const bool cst = xmax == xmin;
  xmin = cst ? fminf(xmin, 0.0f) : xmin;
  xmax = cst ? fmaxf(xmax, 0.0f) : xmax;
  const float range = __fsub_rn(xmax, xmin);  // 0 exactly when xmax == xmin (gradual underflow)
  float s32 = div_rn(range, __fsub_rn(Q<BITS>::qmax, Q<BITS>::qmin), inv_levels<BITS>());
  // binary16 holds every integer only up to 2048: a narrow group far from zero gets the
  // wider scale max|x| / (2048 - 2^BITS), so that |x / scale| <= 2048 - 2^BITS and the
  // zero point (|zp| <= 2048 - 2^(BITS-1)) is stored exactly
  const float s_far = div_rn(fmaxf(fabsf(xmin), fabsf(xmax)), (float)(2048 - (1 << BITS)), inv_far<BITS>());
  s32 = fmaxf(s32, s_far);
  s_h = range == 0.0f ? __float2half_rn(1.0f) : __float2half_ru(s32);  // all zeros: scale 1
  s = __half2float(s_h);
  rs = __frcp_rn(s);
  const float z = __fsub_rn(Q<BITS>::qmin, rintf(div_rn(xmin, s, rs)));  // an integer, |z| <= 2048
  z_h = __float2half_rn(z);
  zp = __half2float(z_h);
}

// Symmetric scale ("KV Cache Quantization — 8-bit and 4-bit", § Symmetric vs asymmetric:
// zero point 0, integer range centred on real zero) from the exact binary32 max|x| of
// binary16 inputs: s_h = binary16 round up of max|x| / 127 (RN(1/127) = 0x3C010204; the
// quotient is correctly rounded, see div_rn), scale 1 for an all-zero vector; s and
// rs = RN(1/s) as binary32. The code is then quant_code<8>(x, s, rs, 128) (zero point 0).
__device__ __forceinline__ void sym_params8(float amax, __half& s_h, float& s, float& rs) {
  if (amax == 0.0f) s_h = __float2half_rn(1.0f);
  else s_h = __float2half_ru(div_rn(amax, 127.0f, __int_as_float(0x3C010204)));
  s = __half2float(s_h);
  rs = __frcp_rn(s);
}

// Code u = clamp(rint(x/s) + zp, q_min, q_max) - q_min of x in a group with binary16
// scale s (rs = RN(1/s)); zpu = zp - q_min (an integer), so the clamp bounds become
// [0, 2^b - 1]. rint rounds half to even; the integer steps are exact, so this equals the
// binary32 formula.
template <int BITS>
__device__ __forceinline__ uint32_t quant_code(float x, float s, float rs, int zpu) {
  const int q = __float2int_rn(div_rn(x, s, rs));
  return (uint32_t)max(__viaddmin_s32(q, zpu, (1 << BITS) - 1), 0);
}

__device__ __forceinline__ void load4(const __half* p, float* x) {
  const uint2 raw = *reinterpret_cast<const uint2*>(p);
  const __half2 a = *reinterpret_cast<const __half2*>(&raw.x);
  const __half2 b = *reinterpret_cast<const __half2*>(&raw.y);
  x[0] = __low2float(a);
  x[1] = __high2float(a);
  x[2] = __low2float(b);
  x[3] = __high2float(b);
}

// Channel stored at value-row position p (inverse of pos(c) = 16*(c%8) + 2*(c/16) + (c/8)%2, d = 128).
__device__ __forceinline__ int v_channel_of_pos(int p) {
  const int g = p >> 4, i = p & 15;
  return 16 * (i >> 1) + 8 * (i & 1) + g;
}

// One warp quantizes one value row (binary16, 128 channels; lane l holds channels
// [4l, 4l+4)) per group of Gv channels, writes its scale and zero point of group j to
// rec[4j] and rec[4j + 2] (rec: the token's half of its pair's metadata records) and its
// codes, in stored-position order, into half `half_sel` of the 16-bit units of its pair
// row. codes_s: 128 bytes of warp-private shared memory.
// SYM: the symmetric per-token scheme (BITS 8, one group of d channels, zero point 0).
template <int BITS, bool SYM = false>
__device__ __forceinline__ void quantize_value_row(const __half* v_row, uint16_t* pair_row, int half_sel, __half* rec,
                                                   int Gv, int lane, uint8_t* codes_s) {
  float x[4];
  load4(v_row + 4 * lane, x);
  const int lanes_per_group = Gv / 4;  // 8, 16 or 32
  __half s_h, z_h;
  float s, rs, zp;
  if constexpr (SYM) {
    float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
    for (int off = 1; off < 32; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
    sym_params8(a, s_h, s, rs);
    z_h = __float2half_rn(0.0f);
    zp = 0.0f;
  } else {
    float mn = fminf(fminf(x[0], x[1]), fminf(x[2], x[3]));
    float mx = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    for (int off = 1; off < lanes_per_group; off <<= 1) {
      mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    }
    group_params<BITS>(mn, mx, s_h, z_h, s, rs, zp);
  }
  if (lane % lanes_per_group == 0) {
    rec[4 * (lane / lanes_per_group)] = s_h;
    rec[4 * (lane / lanes_per_group) + 2] = z_h;
  }
  const int zpu = (int)zp - (int)Q<BITS>::qmin;
#pragma unroll
  for (int e = 0; e < 4; ++e) codes_s[4 * lane + e] = (uint8_t)quant_code<BITS>(x[e], s, rs, zpu);
  __syncwarp();
  constexpr int PER_UNIT = 16 / BITS;
  constexpr int UNITS = kHeadDim * BITS / 16;
  for (int k = lane; k < UNITS; k += 32) {
    uint32_t unit = 0;
#pragma unroll
    for (int i = 0; i < PER_UNIT; ++i) unit |= (uint32_t)codes_s[v_channel_of_pos(k * PER_UNIT + i)] << (i * BITS);
    pair_row[2 * k + half_sel] = (uint16_t)unit;
  }
  __syncwarp();
}

// The 64th smallest (index 63 in ascending order) of the warp's 128 keys, lane l holding
// elements 4l .. 4l + 3. A bitonic sorting network (Batcher) sorts the two halves of 64
// positions, lanes 0-15 ascending and lanes 16-31 descending, which together form a
// bitonic sequence; one compare-exchange at distance 64 (the network's next step) then
// leaves the 64 smallest keys in positions 0-63, and their maximum is the 64th smallest:
// the rest of the last merge stage is not needed. Compare-exchanges at distance 1 and 2
// run inside a lane, at distance 4j across lanes l and l ^ j with a shuffle.
// PAIR: every word holds the 16-bit keys of two rows (low and high halves), handled at
// once with 16x2 SIMD min/max (the network does not depend on the data); the result
// holds both rows' 64th smallest keys.
template <bool PAIR = false>
__device__ __forceinline__ uint32_t kmin(uint32_t a, uint32_t b) { return PAIR ? __vminu2(a, b) : min(a, b); }
template <bool PAIR = false>
__device__ __forceinline__ uint32_t kmax(uint32_t a, uint32_t b) { return PAIR ? __vmaxu2(a, b) : max(a, b); }

template <bool PAIR = false>
__device__ __forceinline__ uint32_t sorted_key_63(const uint32_t (&key_in)[4], int lane) {
  uint32_t a[4] = {key_in[0], key_in[1], key_in[2], key_in[3]};
#pragma unroll
  for (int k = 2; k <= 64; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= 4) {
        const int lj = j >> 2;                         // partner lane distance
        const bool up = (lane & (k >> 2)) == 0;        // this block sorts ascending
        const bool low = (lane & lj) == 0;             // this lane holds the lower positions
        const bool keep_min = (up == low);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t o = __shfl_xor_sync(0xffffffffu, a[e], lj);
          a[e] = keep_min ? kmin<PAIR>(a[e], o) : kmax<PAIR>(a[e], o);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e & j) continue;                         // e is the lower position of the pair (e, e + j)
          const int i = 4 * lane + e;
          const bool up = (i & k) == 0;
          const uint32_t lo = kmin<PAIR>(a[e], a[e + j]), hi = kmax<PAIR>(a[e], a[e + j]);
          a[e] = up ? lo : hi;
          a[e + j] = up ? hi : lo;
        }
      }
    }
  }
  // distance 64: lanes 0-15 keep the minima of positions i and i + 64 (lane l ^ 16), the
  // 64 smallest keys; their maximum over the 16 lanes (lanes 16-31 reduce their own half)
  uint32_t m = 0u;
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint32_t lo = kmin<PAIR>(a[e], __shfl_xor_sync(0xffffffffu, a[e], 16));
    m = e ? kmax<PAIR>(m, lo) : lo;
  }
#pragma unroll
  for (int off = 8; off > 0; off >>= 1) m = kmax<PAIR>(m, __shfl_xor_sync(0xffffffffu, m, off));
  return __shfl_sync(0xffffffffu, m, 0);
}

// Order-preserving 16-bit keys of binary16 bit patterns (negative values bit-inverted,
// positive ones with the sign bit set); -0 and +0 get distinct keys, which leaves
// |x - median| unchanged.
__device__ __forceinline__ void order_keys(const uint32_t (&xb)[4], uint32_t (&key)[4]) {
#pragma unroll
  for (int e = 0; e < 4; ++e) key[e] = (xb[e] & 0x8000u) ? (~xb[e] & 0xFFFFu) : (xb[e] | 0x8000u);
}
__device__ __forceinline__ float value_of_key(uint32_t k) {
  const uint32_t bits = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
  return __half2float(__ushort_as_half((unsigned short)bits));
}

// The kout entries of a key row (xb as in split_row_outliers) farthest from `med` in
// binary32 |x - med|, in order of decreasing distance, ties to the lower channel, to
// entries[0 .. kout) as channel | binary16 << 16 (written by the lane that holds them),
// marked in `taken`.
__device__ __forceinline__ void take_farthest(const uint32_t (&xb)[4], float med, bool (&taken)[4], uint32_t* entries,
                                              int kout, int lane) {
  // distances are non-negative binary32 values, which order like their bit patterns: one
  // warp max of the bits per round, then the lowest lane holding that distance (its
  // channels are the lowest), then that lane's lowest such channel
  uint32_t db[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    taken[e] = false;
    db[e] = __float_as_uint(fabsf(__fsub_rn(__half2float(__ushort_as_half((unsigned short)xb[e])), med)));
  }
  for (int r = 0; r < kout; ++r) {
    uint32_t mine = 0u;
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (!taken[e]) mine = max(mine, db[e] + 1u);  // + 1: an untaken +0 distance still beats a taken entry
    const uint32_t best = __reduce_max_sync(0xffffffffu, mine);
    const uint32_t owners = __ballot_sync(0xffffffffu, mine == best);
    if (lane == __ffs(owners) - 1) {
#pragma unroll
      for (int e = 0; e < 4; ++e)
        if (!taken[e] && db[e] + 1u == best) {
          taken[e] = true;
          entries[r] = (uint32_t)(4 * lane + e) | (xb[e] << 16);
          break;
        }
    }
  }
}

// Dense-and-sparse split of one key row ("Sub-8-Bit KV Cache Quantization Is Not a Free
// Lever for an RDNA4 Agent Swarm", § What the low-bit numbers actually cost: per-vector
// dense-and-sparse quantization). The warp holds the row's 128 binary16 values, lane l the
// bit patterns xb[0..3] of channels [4l, 4l+4); the row's kout entries farthest from its
// lower median (the 64th smallest value) in binary32 |x - median|, in order of decreasing
// distance, ties to the lower channel, go to entries[0 .. kout) as channel | binary16 << 16
// (written by the lane that holds them) and are marked in `taken` (the caller replaces them
// by +0). SORT picks how the lower median is found: a bitonic sort of the row's 128 order
// keys (fewer instructions; the append kernels) or a radix select with warp ballots (the
// fused decode step); both give the exact 64th smallest value.
template <bool SORT>
__device__ __forceinline__ void split_row_outliers(const uint32_t (&xb)[4], bool (&taken)[4], uint32_t* entries,
                                                   int kout, int lane) {
  uint32_t key[4];
  order_keys(xb, key);
  uint32_t prefix = 0;
  if constexpr (SORT) {
    prefix = sorted_key_63(key, lane);
  } else {  // most-significant-bit-first radix select of rank 63, one ballot per key and bit
    int rank = 63;
#pragma unroll
    for (int bit = 15; bit >= 0; --bit) {
      const uint32_t above = (0xFFFFu << (bit + 1)) & 0xFFFFu;  // the bits already decided
      int n0 = 0;
#pragma unroll
      for (int e = 0; e < 4; ++e)
        n0 += __popc(__ballot_sync(0xffffffffu, ((key[e] ^ prefix) & above) == 0u && ((key[e] >> bit) & 1u) == 0u));
      if (rank >= n0) {
        rank -= n0;
        prefix |= 1u << bit;
      }
    }
  }
  take_farthest(xb, value_of_key(prefix), taken, entries, kout, lane);
}

// split_row_outliers (sorting) of two key rows held by the warp at once: their order keys
// share one sort (PAIR), then each row takes its own farthest entries.
__device__ __forceinline__ void split_two_rows_outliers(const uint32_t (&xa)[4], const uint32_t (&xb)[4],
                                                        bool (&taken_a)[4], bool (&taken_b)[4], uint32_t* entries_a,
                                                        uint32_t* entries_b, int kout, int lane) {
  uint32_t ka[4], kb[4], kp[4];
  order_keys(xa, ka);
  order_keys(xb, kb);
#pragma unroll
  for (int e = 0; e < 4; ++e) kp[e] = ka[e] | (kb[e] << 16);
  const uint32_t med2 = sorted_key_63<true>(kp, lane);
  take_farthest(xa, value_of_key(med2 & 0xFFFFu), taken_a, entries_a, kout, lane);
  take_farthest(xb, value_of_key(med2 >> 16), taken_b, entries_b, kout, lane);
}

// One warp quantizes one key row of the symmetric per-token scheme (binary16, 128
// channels; lane l holds channels [4l, 4l+4)): its binary16 scale to *scale_out and its
// 8-bit codes, in channel order, to key_row. With kout > 0 the row's kout farthest
// entries are split off first (split_row_outliers) and replaced by 0 before the scale
// is taken.
// The symmetric int8 codes and binary16 scale of one dense key row held by the warp (lane
// l: channels [4l, 4l+4) as binary32 values), to key_row (channel order) and *scale_out.
__device__ __forceinline__ void quantize_sym_row(const float (&x)[4], uint8_t* key_row, __half* scale_out, int lane) {
  float a = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
  for (int off = 1; off < 32; off <<= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
  __half s_h;
  float s, rs;
  sym_params8(a, s_h, s, rs);
  uint32_t w = 0;
#pragma unroll
  for (int e = 0; e < 4; ++e) w |= quant_code<8>(x[e], s, rs, 128) << (8 * e);
  reinterpret_cast<uint32_t*>(key_row)[lane] = w;
  if (lane == 0) *scale_out = s_h;
}

template <bool SORT = false>
__device__ __forceinline__ void quantize_key_row_sym(const __half* k_row, uint8_t* key_row, __half* scale_out,
                                                     uint32_t* entries, int kout, int lane) {
  float x[4];
  load4(k_row + 4 * lane, x);
  if (kout > 0) {
    const uint2 raw = *reinterpret_cast<const uint2*>(k_row + 4 * lane);
    const uint32_t xb[4] = {raw.x & 0xFFFFu, raw.x >> 16, raw.y & 0xFFFFu, raw.y >> 16};
    bool taken[4];
    split_row_outliers<SORT>(xb, taken, entries, kout, lane);
#pragma unroll
    for (int e = 0; e < 4; ++e)
      if (taken[e]) x[e] = 0.0f;
  }
  quantize_sym_row(x, key_row, scale_out, lane);
}

}  // namespace quant
}  // namespace kvq
