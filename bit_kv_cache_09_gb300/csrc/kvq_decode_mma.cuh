// kvq_decode_mma.cuh — split-K decode attention with tensor-core products over the
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
//           A = folded query x = q*s (rows: query heads, hi and lo binary16 halves,
//               formed with packed half multiply/fma after power-of-two scaling of
//               the query row and of the group's scales), B = key codes. The bias
//               term is one more MMA tile per key group whose B columns hold ones
//               and the group's zero points.
//   output  O[c][i] = sum_t u_tc (p_it s_tj) + sum_t p_it s_tj (q_min - zp_tj)
//           A = value codes (rows: channels), B = weights w = p*s (hi and lo halves,
//           packed half arithmetic). The zero-point sums sum_t w and sum_t zp_t w run
//           as one more MMA tile per value group (A rows: ones and zero points).
//
// Codes enter the MMA as binary16 subnormals: the 16-bit pattern u IS the value
// u * 2^-24, so unpacking is a mask (and a byte permute for 8-bit codes), and the
// 2^24 factor is restored on the binary32 results. Packed layouts are chosen so that
// every lane's fragment comes from one contiguous chunk (see include/kvq.h): key row
// chunk j of a lane holds channels [32j, 32j+32); value pair-row chunk g holds
// channels {16m + g, 16m + g + 8}.
//
// Staging: every warp streams its own contiguous run of 32-token iterations through a
// ring of NS shared-memory stages filled by per-lane 16-byte asynchronous copies
// (cp.async, completion counted on one mbarrier per stage), with bounded waits. A CTA
// (4 warps) merges its warps; splits merge through the workspace (last CTA, atomic
// ticket) or, for small grids, through distributed shared memory of a cluster.
#pragma once

#include <cooperative_groups.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "kvq_common.cuh"
#include "kvq_kernels.h"
#include "kvq_merge.cuh"
#include "kvq_quantizer.cuh"

namespace kvq {
namespace mma {

namespace cg = cooperative_groups;

constexpr int kSlab = 16;

__device__ __forceinline__ void mma16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                         uint32_t b1) {
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The same product with a zero accumulator input (first k-step of a tile).
__device__ __forceinline__ void mma16816_z(float* d, uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                                           uint32_t b1) {
  const float z = 0.0f;
  asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%10,%10,%10,%10};\n"
      : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
      : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(z));
}

// Transpose of an 8x8 matrix of 16-bit elements held one row pair per lane (lane l:
// row l/4, columns 2(l%4), 2(l%4)+1), which is the accumulator layout of an 8-row slice
// of an m16n8 tile packed to binary16; the result is the k16 x n8 operand layout.
__device__ __forceinline__ uint32_t movmatrix_t(uint32_t x) {
  uint32_t d;
  asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(x));
  return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(0u), "r"(sel));
  return d;
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t h2_bits(__half2 h) { return *reinterpret_cast<uint32_t*>(&h); }

// Byte permute of two words (selector nibbles 0..7 pick bytes of {b, a}).
__device__ __forceinline__ uint32_t prmt2(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

// Packed binary16 arithmetic with one IEEE rounding each (.rn keeps the compiler from
// contracting a product into a later add).
__device__ __forceinline__ uint32_t hmul2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
__device__ __forceinline__ uint32_t hmax2(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// a*b split into binary16 halves: hi = fl(a*b), lo = fl(a*b - hi) (the residual is exact
// when it is representable, so hi + lo carries ~22 bits of the product).
__device__ __forceinline__ uint32_t hneg2(uint32_t a) {
  uint32_t d;
  asm("neg.f16x2 %0, %1;" : "=r"(d) : "r"(a));
  return d;
}
__device__ __forceinline__ void hmul2_split(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
  hi = hmul2(a, b);
  lo = hfma2(a, b, hneg2(hi));
}
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }  // e in [-126, 127]

constexpr uint32_t kOne2 = 0x3C003C00u;  // half2(1, 1)

// Words of one lane's chunk of a key row / value pair row (rowK/4 bytes).
template <int BITS>
struct Chunk {
  static constexpr int WORDS = BITS * 128 / 8 / 4 / 4;  // 8, 4, 2
};

// Key codes: pair pi (0..15) of lane chunk j -> half2 of channels (ca, cb) as binary16
// subnormals. A code may be left shifted inside its 16-bit half as long as the pattern
// stays below 0x400 (the subnormal range): the value is then u * 2^-24 * k_scale(pi),
// and the matching query entries are divided by k_scale(pi). This saves the shifts.
template <int BITS>
__device__ __forceinline__ uint32_t k_pair(const uint32_t* w, int pi) {
  if (BITS == 8) return prmt(w[pi >> 1], (pi & 1) ? 0x4342u : 0x4140u);
  if (BITS == 4) {
    const int s = pi & 3;
    const uint32_t x = (s < 2) ? w[pi >> 2] : (w[pi >> 2] >> 8);
    return x & ((s & 1) ? 0x00F000F0u : 0x000F000Fu);
  }
  const int s = pi & 7;
  const uint32_t x = (s < 5) ? w[pi >> 3] : (w[pi >> 3] >> 10);
  return x & (0x00030003u << (2 * (s < 5 ? s : s - 5)));
}

// Scale k_pair leaves on pair pi (a power of two; 1 for 8-bit codes).
template <int BITS>
__device__ __forceinline__ constexpr float k_scale(int pi) {
  return BITS == 8 ? 1.0f
                   : (BITS == 4 ? (((pi & 3) & 1) ? 16.0f : 1.0f)
                                : (float)(1 << (2 * ((pi & 7) < 5 ? (pi & 7) : (pi & 7) - 5))));
}

// half2 bit pattern of k_scale(pi) * 2^-8 (a normal binary16 power of two).
template <int BITS>
__device__ __forceinline__ constexpr uint32_t kc_bits(int pi) {
  const int sh = BITS == 8 ? 0 : (BITS == 4 ? 4 * (pi & 1) : 2 * ((pi & 7) < 5 ? (pi & 7) : (pi & 7) - 5));
  return (uint32_t)(sh + 7) << 10 | (uint32_t)(sh + 7) << 26;
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
  return k_pair_ca<BITS>(pi) + (BITS == 8 ? 1 : (BITS == 4 ? 4 : 8));
}

// Value codes: position i (0..15) of lane chunk g in a pair row -> half2(token 2p, token 2p+1),
// left in place inside the 16-bit halves like k_pair (scale v_scale(i), undone per channel).
template <int BITS>
__device__ __forceinline__ uint32_t v_pair(const uint32_t* w, int i) {
  if (BITS == 8) return prmt(w[i >> 1], (i & 1) ? 0x4341u : 0x4240u);
  if (BITS == 4) {
    const int s = i & 3;
    const uint32_t x = (s < 2) ? w[i >> 2] : (w[i >> 2] >> 8);
    return x & ((s & 1) ? 0x00F000F0u : 0x000F000Fu);
  }
  const int s = i & 7;
  const uint32_t x = (s < 5) ? w[i >> 3] : (w[i >> 3] >> 10);
  return x & (0x00030003u << (2 * (s < 5 ? s : s - 5)));
}

template <int BITS>
__device__ __forceinline__ constexpr float v_scale(int i) {
  return k_scale<BITS>(i);
}

// One stage = one iteration of 32 tokens (two 16-token halves):
//   [key codes 32*rowK][value pair rows 32*rowV][value meta 32*4*NVG B][key meta]
// where the key meta is one key group's (scale, zero point) per channel (512 B), or in
// the symmetric per-token scheme (SYM) the 32 tokens' binary16 key scales (64 B).
// NW warps per CTA each own a ring of NS stages. After the loop the rings are reused
// for the merges: per-warp partials (o, m, l, beta), the CTA partial read by the
// cluster merge (cm, cl, co), then the scratch of the workspace merge.
template <int BITS, int VBITS, int NVG, int NW, bool SYM = false, bool OUTL = false>
struct Stage {
  static constexpr int KB = 32 * BITS * 128 / 8;   // key codes of 32 tokens
  static constexpr int VB = 32 * VBITS * 128 / 8;  // value codes of 32 tokens
  static constexpr int VM = 32 * 4 * NVG;         // value meta of 32 tokens
  // one key group's meta, or 32 key scales; with isolated key entries (OUTL) followed by the
  // 32 tokens' entry lists (up to 4 entries of 4 bytes each) at offset KE
  static constexpr int KE = SYM ? 64 : 512;
  static constexpr int KM = KE + (OUTL ? 512 : 0);
  static constexpr int BYTES = KB + VB + VM + KM;
  static constexpr int NS = BITS == 2 ? 3 : 2;
  static constexpr int WARP_BYTES = NS * BYTES;
  static constexpr int EP_M = NW * kMaxGqa * kHeadDim * 4;
  static constexpr int EP_L = EP_M + NW * kMaxGqa * 4;
  static constexpr int EP_BETA = EP_L + NW * kMaxGqa * 4;
  static constexpr int EP_CM = EP_BETA + NW * kMaxGqa * NVG * 4;
  static constexpr int EP_SCRATCH = (EP_CM + (2 * kMaxGqa + kMaxGqa * kHeadDim) * 4 + 15) / 16 * 16;
  static constexpr int kEpilogueBytes = EP_SCRATCH + 4 * kMergeScratchFloats;
  // isolated key entries: per warp a [32 tokens][kMaxGqa + 1] binary32 table of the sparse
  // score terms, after the stage rings (used in the loop only, like the rings)
  static constexpr int SP = NW * WARP_BYTES;
  static constexpr int SP_ROW = kMaxGqa + 1;
  static constexpr int LOOP_BYTES = SP + (OUTL ? NW * 32 * SP_ROW * 4 : 0);
  static constexpr int SMEM = LOOP_BYTES > kEpilogueBytes ? LOOP_BYTES : kEpilogueBytes;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }


// A stage barrier completes a phase when all 32 lanes of the warp have seen their
// copies of the stage land (cp.async.mbarrier.arrive.noinc, one arrival per lane).
__device__ __forceinline__ void mbar_init(uint32_t bar) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], 32;" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n .reg .pred P;\n mbarrier.try_wait.parity.shared::cta.b64 P, [%1], %2;\n selp.u32 %0, 1, 0, P;\n}\n"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for a stage's copies; gives up after limit_ns of %globaltimer (returns false)
// instead of spinning forever. A limit of 0 gives up at once, without looking.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (limit_ns == 0) return false;
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_ns();
  while (true) {
    for (int k = 0; k < 64; ++k)
      if (mbar_try_wait(bar, parity)) return true;
    if (global_ns() - t0 > limit_ns) return false;
  }
}

constexpr uint64_t kDrainWaitNs = 2000000000ull;  // draining the copies in flight after a failed wait

// 16-byte asynchronous global -> shared copy (L2 only), per thread.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// Arrive on `bar` once this thread's earlier cp.async copies have completed.
__device__ __forceinline__ void cp_async_arrive(uint32_t bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(bar) : "memory");
}

template <int BITS>
__device__ __forceinline__ void lds_chunk(const uint8_t* p, uint32_t* w) {
  if (BITS == 8) {
    const uint4 a = reinterpret_cast<const uint4*>(p)[0];
    const uint4 b = reinterpret_cast<const uint4*>(p)[1];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w; w[4] = b.x; w[5] = b.y; w[6] = b.z; w[7] = b.w;
  } else if (BITS == 4) {
    const uint4 a = reinterpret_cast<const uint4*>(p)[0];
    w[0] = a.x; w[1] = a.y; w[2] = a.z; w[3] = a.w;
  } else {
    const uint2 a = reinterpret_cast<const uint2*>(p)[0];
    w[0] = a.x; w[1] = a.y;
  }
}

// value meta of token pair (tl, tl + 1), tl even: per group the half2 of the two scales,
// then the half2 of the two zero points (2 * NVG half2)
template <int NVG>
__device__ __forceinline__ void lds_vmeta(const __half2* p, __half2* m) {
  if (NVG == 1) {
    const uint2 a = *reinterpret_cast<const uint2*>(p);
    m[0] = *reinterpret_cast<const __half2*>(&a.x);
    m[1] = *reinterpret_cast<const __half2*>(&a.y);
  } else if (NVG == 2) {
    const uint4 a = *reinterpret_cast<const uint4*>(p);
    m[0] = *reinterpret_cast<const __half2*>(&a.x);
    m[1] = *reinterpret_cast<const __half2*>(&a.y);
    m[2] = *reinterpret_cast<const __half2*>(&a.z);
    m[3] = *reinterpret_cast<const __half2*>(&a.w);
  } else {
    const uint4 a = reinterpret_cast<const uint4*>(p)[0];
    const uint4 b = reinterpret_cast<const uint4*>(p)[1];
    m[0] = *reinterpret_cast<const __half2*>(&a.x);
    m[1] = *reinterpret_cast<const __half2*>(&a.y);
    m[2] = *reinterpret_cast<const __half2*>(&a.z);
    m[3] = *reinterpret_cast<const __half2*>(&a.w);
    m[4] = *reinterpret_cast<const __half2*>(&b.x);
    m[5] = *reinterpret_cast<const __half2*>(&b.y);
    m[6] = *reinterpret_cast<const __half2*>(&b.z);
    m[7] = *reinterpret_cast<const __half2*>(&b.w);
  }
}

// Resident CTAs per SM the register budget is sized for: 4 at 128 registers (r <= 4),
// 3 at 168 (r <= 8: its hi and lo P.V products share one accumulator tile, which keeps
// the kernel within 168 registers without spills).
template <int NT>
constexpr int min_blocks() {
  return NT == 1 ? 4 : 3;
}

// SYM: the symmetric per-token int8 scheme ("KV Cache Quantization — 8-bit and 4-bit",
// § Symmetric vs asymmetric; one scale per token, "Sub-8-Bit KV Cache Quantization Is
// Not a Free Lever for an RDNA4 Agent Swarm", § The RDNA4 kernel angle): no query fold;
// the raw query meets the exact key codes on the tensor cores and the score of token t
// is s_t * (2^24 acc + q_min * sum_c q_c) in softmax units; values as in the
// asymmetric scheme with one group and zero point 0.
// BITS, VBITS: key and value code widths; NT: PV weight tiles per k-step (1: r <= 4, hi/lo
// halves share one tile; 2: r <= 8, a hi and a lo tile accumulated into the same output
// tile); NVG: value groups per token (d / Gv); NW: warps per
// CTA (4; 5 or 8 for small cluster-merged grids, where few CTAs per SM are resident
// anyway and more warps shorten the busiest warp's run of iterations; the 5-warp CTA
// keeps two CTAs per SM).
// MIXED: the grid is a mixed plan's one-dimensional list of CTAs (4-warp CTAs only).
template <int BITS, int VBITS, int NT, int NVG, int NW, bool SYM = false, bool OUTL = false, bool MIXED = false>
__global__ void __launch_bounds__(NW * 32, NW == 4 ? min_blocks<NT>() : (NW == 5 ? 2 : 1)) decode_mma_kernel(DecodeParams p) {
  constexpr int kWarps = NW;
  using St = Stage<BITS, VBITS, NVG, NW, SYM, OUTL>;
  constexpr int NS = St::NS;
  constexpr int kTok = 32;  // tokens per iteration
  constexpr float qmin = -(float)(1 << (BITS - 1));     // keys
  constexpr float qmin_v = -(float)(1 << (VBITS - 1));  // values
  constexpr int CW = Chunk<BITS>::WORDS;
  constexpr int CWV = Chunk<VBITS>::WORDS;
  constexpr int ROW = BITS * 128 / 8;    // bytes per key row
  constexpr int ROWV = VBITS * 128 / 8;  // bytes per value row
  constexpr float kTwo24 = 16777216.0f;
  extern __shared__ __align__(128) uint8_t smem[];
  __shared__ __align__(8) uint64_t bars[kWarps][NS];
  __shared__ __align__(16) float q_s[kMaxGqa][kHeadDim];
  // query row i in key-pair order of lane chunk c, pre-divided by k_scale and scaled
  // by 2^qe_s[i] (so that |entry| < 2^8), as binary16 pairs
  __shared__ __align__(16) uint32_t q2_s[SYM ? 1 : kMaxGqa][4][16];  // not used by per-token key scales
  __shared__ int qe_s[kMaxGqa];
  __shared__ float qsum_s[kMaxGqa];  // SYM: sum_c q_c of every query row
  // padded rows: no bank conflicts. SYM keeps only the hi words (the lo rows of its A
  // fragments are zero): 16 words per row, 18 with the padding
  constexpr int kQA = SYM ? 18 : 36;
  __shared__ __align__(16) uint32_t qa_s[(NT == 1) ? 1 : kWarps][(NT == 1) ? 1 : 32][kQA];
  // r <= 4 (NT == 1): key codes are the A operand (token rows) and the query the B operand,
  // column n = 2q + h holding query q's hi (h = 0) or lo (h = 1) halves; one padded row of
  // B fragments per (column, lane chunk): word 2ks + e is fragment register e of k-step ks
  constexpr int kQB = 20;
  __shared__ __align__(16) uint32_t qb_s[(NT == 1) ? kWarps : 1][8][4][kQB];
  // fused step: codes of the new value row on their way into the pair row. Not the stage
  // rings: with early prefetch their first stages are already being filled.
  __shared__ __align__(16) uint8_t append_s[kHeadDim];

  // this CTA's (batch row, kv head) pair, split, split length and the number of parts its
  // pair merges through the workspace: from the grid (n_split, H, B), or from a mixed plan's
  // list (the first pairs_hi pairs in n_hi splits of chunk_hi tokens, the rest in n_hi - 1
  // splits of chunk_lo tokens)
  int split_m = 0, h_m = 0, b_m = 0, parts_m = 0, chunk_m = 0;
  if constexpr (MIXED) {
    const int c = (int)blockIdx.x, ctas_hi = p.pairs_hi * p.n_hi;
    int pair;
    if (c < ctas_hi) {
      pair = c / p.n_hi;
      split_m = c - pair * p.n_hi;
      parts_m = p.n_hi;
      chunk_m = (int)p.chunk_hi;
    } else {
      const int n_lo = p.n_hi - 1, c2 = c - ctas_hi;
      pair = p.pairs_hi + c2 / n_lo;
      split_m = c2 - (c2 / n_lo) * n_lo;
      parts_m = n_lo;
      chunk_m = (int)p.chunk_lo;
    }
    b_m = pair / p.H;
    h_m = pair - b_m * p.H;
  }
  const int split = MIXED ? split_m : (int)blockIdx.x;
  const int h = MIXED ? h_m : (int)blockIdx.y, b = MIXED ? b_m : (int)blockIdx.z;
  const int n_parts = MIXED ? parts_m : p.n_parts;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g = lane >> 2, j = lane & 3;
  const int r = p.r;
  const int qi = (NT == 1) ? ((g & 3) % r) : (g % r);  // query head of QK row g / PV column g
  const int64_t slice = (int64_t)b * p.H + h;
  const int64_t qrow0 = (int64_t)b * p.H * r + (int64_t)h * r;

  const int T = (int)p.T, Tq = (int)p.Tq;
  const int t_begin = split * (MIXED ? chunk_m : (int)p.chunk);  // chunk is a multiple of 32
  const int t_end = min(t_begin + (MIXED ? chunk_m : (int)p.chunk), T);
  const int n_it = max(0, (t_end - t_begin + kTok - 1) / kTok);  // 0 for a trailing empty split
  // balanced contiguous runs of iterations per warp (warp w: [w*n_it/NW, (w+1)*n_it/NW))
  const int it0 = (warp * n_it) / kWarps;
  const int n_mine = ((warp + 1) * n_it) / kWarps - it0;
  const int ts0 = t_begin + it0 * kTok;  // first token of this warp (a multiple of 32)

  uint8_t* wbase = smem + warp * St::WARP_BYTES;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(smem_u32(&bars[warp][s]));
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();

  // sources of the warp's first iteration; iteration i adds 32*i tokens
  const uint8_t* k_src = p.k_codes + slice * p.k_codes_slice + (int64_t)ts0 * ROW;
  const uint8_t* v_src = p.v_codes + slice * p.v_codes_slice + (int64_t)ts0 * ROWV;
  const uint8_t* vm_src = reinterpret_cast<const uint8_t*>(p.v_meta + (slice * p.S_pad + ts0) * NVG);
  const __half2* km_base =
      reinterpret_cast<const __half2*>(reinterpret_cast<const uint8_t*>(p.k_meta) + slice * p.k_meta_slice);
  // SYM: per-token key scales of the warp's first iteration (k_meta holds S_pad per slice)
  const uint8_t* ksc_src = reinterpret_cast<const uint8_t*>(p.k_meta) + slice * p.k_meta_slice + (int64_t)ts0 * 2;
  // isolated key entries: p.kout entries (4 B each) per token after the S_pad key scales
  // (symmetric scheme) or after the key groups' (scale, zero point) pairs
  const uint8_t* kent_src = reinterpret_cast<const uint8_t*>(p.k_meta) + slice * p.k_meta_slice +
                            (SYM ? p.S_pad * 2 : (p.S_pad >> p.log2G) * kHeadDim * 4) + (int64_t)ts0 * p.kout * 4;

  // Copies of the warp's iteration i into stage sidx: every lane moves 16-byte pieces
  // (piece lane + 32c of each block) with cp.async and arrives on the stage barrier
  // when its pieces have landed. Plain per-thread copies keep the issue cost at a
  // few instructions per lane and iteration.
  const uint32_t wbase_s = smem_u32(wbase) + 16 * lane;
  auto issue = [&](int i, int sidx) {
    constexpr int CK = St::KB / 512, CKV = St::VB / 512;  // pieces per lane of the key / value codes
    const int ts = ts0 + i * kTok;
    const uint32_t dst = wbase_s + sidx * St::BYTES;
    const bool quant = ts < Tq;
    const bool newgrp = quant && (i == 0 || (ts & (p.G - 1)) == 0);
    const size_t off = (size_t)i * St::KB + 16 * lane, offv = (size_t)i * St::VB + 16 * lane;
    if (quant) {
#pragma unroll
      for (int c = 0; c < CK; ++c) cp_async16(dst + 512 * c, k_src + off + 512 * c);
    }
#pragma unroll
    for (int c = 0; c < CKV; ++c) cp_async16(dst + St::KB + 512 * c, v_src + offv + 512 * c);
    if (16 * lane < St::VM) cp_async16(dst + St::KB + St::VB, vm_src + (size_t)i * St::VM + 16 * lane);
    if constexpr (SYM && OUTL) {  // pieces 0..3: 32 key scales; then 32 tokens x kout entries (128 kout bytes)
      for (int pc = lane; pc < 4 + 8 * p.kout; pc += 32) {
        const uint32_t dpc = dst + St::KB + St::VB + St::VM + 16 * (pc - lane);  // dst includes 16 * lane
        if (pc < 4) cp_async16(dpc, ksc_src + (size_t)i * 64 + 16 * pc);
        else cp_async16(dpc, kent_src + (size_t)i * 128 * p.kout + 16 * (pc - 4));
      }
    } else if constexpr (SYM) {
      if (lane < 4) cp_async16(dst + St::KB + St::VB + St::VM, ksc_src + (size_t)i * 64 + 16 * lane);
    } else {
      if (newgrp) cp_async16(dst + St::KB + St::VB + St::VM, km_base + ((ts >> p.log2G) << 7) + 4 * lane);
      if constexpr (OUTL) {  // the 32 quantized tokens' entry lists (128 kout bytes; residual keys have none)
        if (quant && lane < 8 * p.kout)
          cp_async16(dst + St::KB + St::VB + St::VM + St::KE, kent_src + (size_t)i * 128 * p.kout + 16 * lane);
      }
    }
    cp_async_arrive(smem_u32(&bars[warp][sidx]));
  };
  // With p.early the warp's first stages are in flight before the wait on the previous
  // kernel, except the stage that holds the new token T-1 of a fused step (its rows are
  // written below, after the wait).
  const bool owner = p.v_new != nullptr && t_begin <= T - 1 && T - 1 < t_end;
  const int i_new = (owner && ts0 <= T - 1) ? (T - 1 - ts0) / kTok : -1;
  if (p.early) {
    for (int i = 0; i < min(NS, n_mine); ++i)
      if (i != i_new) issue(i, i);
  }
  pdl_wait();  // above: shared memory and, with p.early, cache tiles the previous kernel does not write
  // The next kernel of the stream may launch its CTAs once every CTA of this grid is past
  // its wait (so the kernel before this one has finished): they take SM slots as this
  // grid's CTAs exit, rather than after the slowest CTA's loop.
  pdl_allow_dependents();

  // Query rows of this kv head for warp w: rows w, w + NW, ... (lane l: channels
  // [4l, 4l+4)). Without p.early they are loaded before any stage copy is issued: behind
  // the copies of all resident warps they would arrive only after the first stages, and
  // the query fold (below) is on the path to the first iteration.
  constexpr int kRowsPerWarp = (kMaxGqa + kWarps - 1) / kWarps;
  uint2 qraw[kRowsPerWarp];
#pragma unroll
  for (int k = 0; k < kRowsPerWarp; ++k)
    if (warp + k * kWarps < r)
      qraw[k] = *reinterpret_cast<const uint2*>(p.q + (qrow0 + warp + k * kWarps) * kHeadDim + 4 * lane);

  // Fused decode step: the CTA whose range holds the new token T-1 appends it first
  // (value row quantized per group into its half of the pair row, key row into its
  // residual slot); the barrier orders those global writes before the copies.
  if (p.v_new != nullptr && t_begin <= T - 1 && T - 1 < t_end) {
    if (warp == 0) {
      const int t_new = T - 1;
      const int64_t row = (int64_t)b * p.H + h;  // [B][1][H][d]
      uint16_t* pair = reinterpret_cast<uint16_t*>(p.v_codes_w + slice * p.v_codes_slice + (int64_t)(t_new >> 1) * 2 * ROWV);
      quant::quantize_value_row<VBITS, SYM>(p.v_new + row * kHeadDim, pair, t_new & 1,
                                           reinterpret_cast<__half*>(p.v_meta_w) +
                                               (slice * (p.S_pad >> 1) + (t_new >> 1)) * NVG * 4 + (t_new & 1),
                                           p.Gv, lane, append_s);
      if constexpr (SYM) {  // the key row is quantized per token right away (no residual window)
        uint8_t* kmb = reinterpret_cast<uint8_t*>(p.k_meta_w) + slice * p.k_meta_slice;
        quant::quantize_key_row_sym(p.k_new + row * kHeadDim, p.k_codes_w + slice * p.k_codes_slice + (int64_t)t_new * ROW,
                                    reinterpret_cast<__half*>(kmb) + t_new,
                                    reinterpret_cast<uint32_t*>(kmb + p.S_pad * 2) + (int64_t)t_new * p.kout, p.kout, lane);
      } else {
        const uint2 kv = *reinterpret_cast<const uint2*>(p.k_new + row * kHeadDim + 4 * lane);
        *reinterpret_cast<uint2*>(p.k_resid_w + (slice * p.R_eff + t_new % p.R_eff) * kHeadDim + 4 * lane) = kv;
      }
    }
    __syncthreads();
  }
  for (int i = 0; i < min(NS, n_mine); ++i)
    if (!p.early || i == i_new) issue(i, i);

  // Query rows (loaded above): each row goes to q_s (binary32, for residual keys) and, normalised by
  // 2^qe (qmax * 2^qe in [2^7, 2^8)) and divided by k_scale, to q2_s in key-pair order:
  // pair pi of chunk c = l/8 joins channels ca(pi) and cb(pi), which lie in this lane
  // (8-bit codes) or in the lane 1 (4-bit) or 2 (2-bit) above it.
#pragma unroll
  for (int kq = 0; kq < kRowsPerWarp; ++kq) {
    const int i = warp + kq * kWarps;
    if (i >= r) break;
    const uint2 raw = qraw[kq];
    float xq[4];
    {
      const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
      const float2 c2 = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
      xq[0] = a.x; xq[1] = a.y; xq[2] = c2.x; xq[3] = c2.y;
    }
    reinterpret_cast<float4*>(&q_s[i][0])[lane] = make_float4(xq[0], xq[1], xq[2], xq[3]);
    if constexpr (SYM) {
      float qs = (xq[0] + xq[1]) + (xq[2] + xq[3]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) qs += __shfl_xor_sync(0xffffffffu, qs, o);
      if (lane == 0) qsum_s[i] = qs;
    }
    float a = fmaxf(fmaxf(fabsf(xq[0]), fabsf(xq[1])), fmaxf(fabsf(xq[2]), fabsf(xq[3])));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, o));
    const int qe = a > 0.0f ? 7 - (((__float_as_int(a) >> 23) & 0xFF) - 127) : 0;
    if (lane == 0) qe_s[i] = qe;
    if constexpr (!SYM) {  // per-token key scales need no folded query
      const float f = pow2f(qe);  // exact scaling by a power of two
      float v[4], w[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) v[k] = xq[k] * f;
      constexpr int D = BITS == 8 ? 0 : (BITS == 4 ? 1 : 2);  // lane distance of a pair's second channel
#pragma unroll
      for (int k = 0; k < 4; ++k) w[k] = D ? __shfl_down_sync(0xffffffffu, v[k], D) : v[k];
      const int lc = lane & 7, c = lane >> 3;  // lane within its chunk, chunk
      if (BITS == 8) {  // pairs 2lc (channels 4lc, 4lc+1) and 2lc+1 (4lc+2, 4lc+3)
        q2_s[i][c][2 * lc] = h2_bits(__floats2half2_rn(v[0], v[1]));
        q2_s[i][c][2 * lc + 1] = h2_bits(__floats2half2_rn(v[2], v[3]));
      } else if (BITS == 4) {  // even lc: pairs 4m + e join channels 8m + e and 8m + e + 4 (m = lc/2)
        if ((lc & 1) == 0) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float ks = k_scale<BITS>(e);
            q2_s[i][c][2 * lc + e] = h2_bits(__floats2half2_rn(v[e] / ks, w[e] / ks));
          }
        }
      } else {  // lc % 4 < 2: pairs 8m + 4(lc & 1) + k join channels 16m + 4(lc & 1) + k and + 8
        if ((lc & 3) < 2) {
          const int pi0 = 8 * (lc >> 2) + 4 * (lc & 1);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const float ks = (lc & 1) ? k_scale<BITS>(4 + k) : k_scale<BITS>(k);
            q2_s[i][c][pi0 + k] = h2_bits(__floats2half2_rn(v[k] / ks, w[k] / ks));
          }
        }
      }
    }
  }
  __syncthreads();

  // online softmax state of query qi (identical in the 4 lanes of row g)
  float m_run = -__int_as_float(0x7f800000), l_run = 0.0f;
  // PV accumulators: with r <= 4 one n-tile holds the hi (columns 0..3) and lo (4..7)
  // products; with r > 4 the hi and lo products of queries 0..7 accumulate into the same
  // tile through two MMAs (same MMA count as two tiles, half the registers)
  float o[8][4];
#pragma unroll
  for (int mt = 0; mt < 8; ++mt)
#pragma unroll
    for (int e = 0; e < 4; ++e) o[mt][e] = 0.0f;
  // zero-point sums per value group on the tensor cores: in an extra PV tile rows 0..7
  // are ones and rows 8..15 the tokens' zero points, so every lane accumulates
  // sum_t w_t (registers 0, 1) and sum_t zp_t w_t (registers 2, 3) of its two columns
  float bacc[NVG][4];
#pragma unroll
  for (int k = 0; k < NVG; ++k)
#pragma unroll
    for (int e = 0; e < 4; ++e) bacc[k][e] = 0.0f;
  // query of this lane's scores: with r <= 4 the lanes of column pair (2j, 2j+1) score query
  // j; with r > 4 row g scores query g
  const int qj = (NT == 1) ? (j % r) : qi;
  const int qe_mine = qe_s[qj];
  const float qmin_qsum = SYM ? qmin * qsum_s[qj] : 0.0f;  // SYM: q_min * sum_c q_c of the lane's query

  // r > 4: QK A fragments of the current key group (or of the raw query for residual keys)
  // in shared memory, one padded row per (query, lane chunk): word 4ks + e is fragment
  // register e of k-step ks. r <= 4: B fragments of column g (query g / 2, hi or lo
  // halves), row (g, j) of qb_s. Either way a lane folds query qi (= (g & 3) % r for r <= 4)
  // over half hh of its chunk (r <= 4: lanes g and g + 4 split the chunk).
  uint32_t* qa_row = &qa_s[(NT == 1) ? 0 : warp][(NT == 1) ? 0 : lane][0];
  uint32_t* qb_row = &qb_s[(NT == 1) ? warp : 0][(NT == 1) ? g : 0][(NT == 1) ? j : 0][0];
  const int hh = (NT == 1) ? (g >> 2) : 0;  // first half this lane folds
  float qscale = 0.0f, qbias = 0.0f;
  bool resid_frags = false;
  // raw query row of the fragments for residual (and symmetric) keys: r <= 4 column g's query
  const float* qrow = &q_s[(NT == 1) ? ((g >> 1) % r) : qi][32 * j];

  // Folded query of a key group, x_c = q_c s_c, as binary16 hi/lo pairs computed with
  // packed half arithmetic: q2_s holds q_c 2^qe / k_scale, the scales are scaled by 2^Es
  // so that the largest is in [2^7, 2^8) (no overflow, products below 2^16); hi = fl(q s),
  // lo = fl(q s - hi). Pairs 8h .. 8h + 7 of a lane chunk cover its local channels
  // [16h, 16h + 16) for every code width. Sets qscale and qbias of the group.
  auto fold_group = [&](const uint8_t* st) {
    constexpr int NH = (NT == 1) ? 1 : 2;  // halves folded by this lane
    const uint4* mp = reinterpret_cast<const uint4*>(st + St::KB + St::VB + St::VM) + 8 * j;
    uint32_t mw[NH][16];  // (scale, zero point) of the lane's channels of each half it folds
#pragma unroll
    for (int u = 0; u < NH; ++u)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const uint4 v = mp[4 * (hh + u) + k];
        mw[u][4 * k] = v.x; mw[u][4 * k + 1] = v.y; mw[u][4 * k + 2] = v.z; mw[u][4 * k + 3] = v.w;
      }
    uint32_t s2[NH][8];
    uint32_t mx = 0u;
#pragma unroll
    for (int u = 0; u < NH; ++u) {
#pragma unroll
      for (int pl = 0; pl < 8; ++pl)
        s2[u][pl] = prmt2(mw[u][k_pair_ca<BITS>(pl)], mw[u][k_pair_cb<BITS>(pl)], 0x5410u);
      const uint32_t m01 = hmax2(s2[u][0], s2[u][1]), m23 = hmax2(s2[u][2], s2[u][3]);
      const uint32_t m45 = hmax2(s2[u][4], s2[u][5]), m67 = hmax2(s2[u][6], s2[u][7]);
      const uint32_t m = hmax2(hmax2(m01, m23), hmax2(m45, m67));
      mx = (u == 0) ? m : hmax2(mx, m);
    }
    // the group's largest scale over the warp (every channel is folded by some lane);
    // scales are positive: the larger bit pattern is the larger value
    const uint32_t smax = __reduce_max_sync(0xffffffffu, max(mx & 0xFFFFu, mx >> 16));
    const int Es = min(15, 7 - (max((int)(smax >> 10), 1) - 15));  // in [-8, 15]
    const uint32_t pe = (uint32_t)(Es + 15) << 10;
    const uint32_t p2 = pe | (pe << 16);  // half2(2^Es, 2^Es)
    // bias = sum_c x_c (q_min - zp_c) on the tensor cores, from the fragments just
    // computed: an extra key tile whose column 0 is (q_min - zp_c) k_scale 2^-8 (lane
    // g = 0; q_min - zp_c is an integer of magnitude <= 2048, exact in binary16, and
    // k_scale 2^-8 a power of two). With r <= 4, rows g < 4 run on the first half of the
    // channels and rows g >= 4 on the second in the same MMA, so lane g = 4 supplies the
    // second half's column 4 and a query's bias adds rows q (column 0) and q + 4
    // (column 4).
    float bt[4] = {0.0f, 0.0f, 0.0f, 0.0f};
    const bool bsel = g == 0 || (NT == 1 && g == 4);
    const uint32_t nsel = bsel ? 0xBC00BC00u : 0u;  // half2(-1, -1) in the bias columns
    const uint32_t qsel = bsel ? (uint32_t)__half_as_ushort(__float2half_rn(qmin)) * 0x00010001u : 0u;
#pragma unroll
    for (int u = 0; u < NH; ++u) {
      const int h = hh + u;
      const uint4* qp = reinterpret_cast<const uint4*>(&q2_s[qi][j][8 * h]);
#pragma unroll
      for (int k = 0; k < 2; ++k) {  // k-steps 4h + 2k, 4h + 2k + 1
        const uint4 qv = qp[k];
        const uint32_t qq[4] = {qv.x, qv.y, qv.z, qv.w};
        uint32_t f[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) hmul2_split(qq[e], hmul2(s2[u][4 * k + e], p2), f[2 * e], f[2 * e + 1]);
        if constexpr (NT == 1) {  // hi halves of pairs 8h + 4k + e to column 2(g & 3), lo to the next
          uint32_t* cb = &qb_s[warp][2 * (g & 3)][j][8 * h + 4 * k];
          *reinterpret_cast<uint4*>(cb) = make_uint4(f[0], f[2], f[4], f[6]);
          *reinterpret_cast<uint4*>(cb + 4 * kQB) = make_uint4(f[1], f[3], f[5], f[7]);
        } else {
          reinterpret_cast<uint4*>(qa_row)[4 * h + 2 * k] = make_uint4(f[0], f[1], f[2], f[3]);
          reinterpret_cast<uint4*>(qa_row)[4 * h + 2 * k + 1] = make_uint4(f[4], f[5], f[6], f[7]);
        }
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
          uint32_t bz[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int pl = 4 * k + 2 * kk + e;
            const uint32_t z2 = prmt2(mw[u][k_pair_ca<BITS>(pl)], mw[u][k_pair_cb<BITS>(pl)], 0x7632u);
            bz[e] = hmul2(hfma2(z2, nsel, qsel), kc_bits<BITS>(pl));
          }
          mma16816(bt, f[4 * kk], f[4 * kk + 1], f[4 * kk + 2], f[4 * kk + 3], bz[0], bz[1]);
        }
      }
    }
    __syncwarp();
    // lanes j = 0 hold column 0 of rows g (hi) and g + 8 (lo), lanes j = 2 column 4
    const float t0 = bt[0] + bt[2];
    float bsum;
    if (NT == 1) {  // rows q and q + 4 hold query q's two halves of the channels
      const int q = qj;
      bsum = __shfl_sync(0xffffffffu, t0, 4 * q) + __shfl_sync(0xffffffffu, t0, 4 * q + 18);
    } else {
      bsum = __shfl_sync(0xffffffffu, t0, lane & ~3);
    }
    const int E = qe_mine + Es;
    qscale = pow2f(24 - E) * p.scale_log2;
    qbias = bsum * pow2f(8 - E) * p.scale_log2;
  };

  // r <= 4: B fragments of the raw query (binary16, exact) in natural channel pairs, for
  // residual binary16 keys and the symmetric scheme; lo columns are zero.
  auto raw_query_frags_t = [&]() {
    __syncwarp();
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) {
      const float4 qv = reinterpret_cast<const float4*>(qrow)[ks];
      const uint32_t w0 = (g & 1) ? 0u : h2_bits(__floats2half2_rn(qv.x, qv.y));
      const uint32_t w1 = (g & 1) ? 0u : h2_bits(__floats2half2_rn(qv.z, qv.w));
      reinterpret_cast<uint2*>(qb_row)[ks] = make_uint2(w0, w1);
    }
    __syncwarp();
  };

  // r <= 4: scores of iteration i (stage st) as MMA accumulators acc[m-tile][e]: rows are
  // tokens 16 hf + g (e = 0, 1) and 16 hf + 8 + g (e = 2, 3), columns 2j (hi) and 2j + 1
  // (lo) of query j; s = (acc[e] + acc[e + 1]) * sc + bi.
  auto qk_t = [&](int i, const uint8_t* st, float (&acc)[2][4], float& sc, float& bi) {
    const int ts = ts0 + i * kTok;
    if (ts < Tq) {
      if (SYM && i == 0) raw_query_frags_t();
      if (!SYM && (i == 0 || (ts & (p.G - 1)) == 0)) {
        resid_frags = false;
        fold_group(st);
      }
      uint32_t kw[2][2][CW];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) lds_chunk<BITS>(st + (16 * hf + 8 * nt + g) * ROW + j * (ROW / 4), kw[hf][nt]);
#pragma unroll
      for (int k = 0; k < 4; ++k) {  // k-steps 2k, 2k + 1
        const uint4 bq = reinterpret_cast<const uint4*>(qb_row)[k];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int ks = 2 * k + u;
          const uint32_t b0 = u ? bq.z : bq.x, b1 = u ? bq.w : bq.y;
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            const uint32_t a0 = k_pair<BITS>(kw[hf][0], 2 * ks), a1 = k_pair<BITS>(kw[hf][1], 2 * ks);
            const uint32_t a2 = k_pair<BITS>(kw[hf][0], 2 * ks + 1), a3 = k_pair<BITS>(kw[hf][1], 2 * ks + 1);
            if (ks == 0) mma16816_z(acc[hf], a0, a1, a2, a3, b0, b1);
            else mma16816(acc[hf], a0, a1, a2, a3, b0, b1);
          }
        }
      }
    } else if constexpr (!SYM) {  // binary16 residual keys (the symmetric scheme has none)
      if (!resid_frags) {
        resid_frags = true;
        raw_query_frags_t();
        qscale = p.scale_log2;
        qbias = 0.0f;
      }
      const __half* kr = p.k_resid + slice * (int64_t)p.R_eff * kHeadDim;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        // residual slots of tokens [Tq, T) are t - Tq (Tq is a multiple of the window);
        // rows g and g + 8 of the m-tile, the lane's 32 channels, natural pairs
        uint32_t kw[2][16];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const uint4* rp = reinterpret_cast<const uint4*>(kr + (ts - Tq + 16 * hf + 8 * nt + g) * kHeadDim + 32 * j);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = rp[k];  // plain load: the fused step may have written this row
            kw[nt][4 * k] = v.x; kw[nt][4 * k + 1] = v.y; kw[nt][4 * k + 2] = v.z; kw[nt][4 * k + 3] = v.w;
          }
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 bq = reinterpret_cast<const uint4*>(qb_row)[k];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int ks = 2 * k + u;
            const uint32_t b0 = u ? bq.z : bq.x, b1 = u ? bq.w : bq.y;
            if (ks == 0) mma16816_z(acc[hf], kw[0][0], kw[1][0], kw[0][1], kw[1][1], b0, b1);
            else mma16816(acc[hf], kw[0][2 * ks], kw[1][2 * ks], kw[0][2 * ks + 1], kw[1][2 * ks + 1], b0, b1);
          }
        }
      }
    }
    sc = qscale;
    bi = qbias;
  };

  // r > 4: scores of iteration i (stage st) as MMA accumulators, with the (scale, bias) that
  // turn them into log2-unit scores: s = acc * sc + bi.
  auto qk = [&](int i, const uint8_t* st, float (&acc)[2][2][4], float& sc, float& bi) {
    const int ts = ts0 + i * kTok;
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[hf][nt][e] = 0.0f;
    if (ts < Tq) {
      if (SYM && i == 0) {
        // symmetric per-token keys: the raw query (binary16, exact) in natural channel pairs
        __syncwarp();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const float4 qv = reinterpret_cast<const float4*>(qrow)[ks];
          reinterpret_cast<uint2*>(qa_row)[ks] =
              make_uint2(h2_bits(__floats2half2_rn(qv.x, qv.y)), h2_bits(__floats2half2_rn(qv.z, qv.w)));
        }
        __syncwarp();
      }
      if (!SYM && (i == 0 || (ts & (p.G - 1)) == 0)) {
        resid_frags = false;
        fold_group(st);
      }
      uint32_t kw[2][2][CW];
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) lds_chunk<BITS>(st + (16 * hf + 8 * nt + g) * ROW + j * (ROW / 4), kw[hf][nt]);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint4 a;
        if constexpr (SYM) {
          const uint2 a2 = reinterpret_cast<const uint2*>(qa_row)[ks];
          a = make_uint4(a2.x, 0u, a2.y, 0u);
        } else {
          a = reinterpret_cast<const uint4*>(qa_row)[ks];
        }
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
            mma16816(acc[hf][nt], a.x, a.y, a.z, a.w, k_pair<BITS>(kw[hf][nt], 2 * ks),
                     k_pair<BITS>(kw[hf][nt], 2 * ks + 1));
      }
    } else if constexpr (!SYM) {  // binary16 residual keys (the symmetric scheme has none)
      if (!resid_frags) {
        resid_frags = true;  // raw query fragments for binary16 residual keys: natural channel pairs
        __syncwarp();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const float4 qv = reinterpret_cast<const float4*>(qrow)[ks];
          reinterpret_cast<uint4*>(qa_row)[ks] = make_uint4(h2_bits(__floats2half2_rn(qv.x, qv.y)), 0u,
                                                            h2_bits(__floats2half2_rn(qv.z, qv.w)), 0u);
        }
        __syncwarp();
        qscale = p.scale_log2;
        qbias = 0.0f;
      }
      const __half* kr = p.k_resid + slice * (int64_t)p.R_eff * kHeadDim;
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          // residual slots of tokens [Tq, T) are t - Tq (Tq is a multiple of the window)
          const uint4* rp = reinterpret_cast<const uint4*>(kr + (ts - Tq + 16 * hf + 8 * nt + g) * kHeadDim + 32 * j);
          uint32_t kw[16];
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const uint4 v = rp[k];  // plain load: the fused step may have written this row
            kw[4 * k] = v.x; kw[4 * k + 1] = v.y; kw[4 * k + 2] = v.z; kw[4 * k + 3] = v.w;
          }
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint4 a = reinterpret_cast<const uint4*>(qa_row)[ks];
            mma16816(acc[hf][nt], a.x, a.y, a.z, a.w, kw[2 * ks], kw[2 * ks + 1]);
          }
        }
    }
    sc = qscale;
    bi = qbias;
  };

  // P.V of one stage from the binary16 softmax weights ph[hf][e] of the lane's B column (token
  // pairs (2j, 2j+1), e = 0, and (8+2j, 9+2j), e = 1, of each 16-token half hf): weights
  // w = p * s per value group as binary16 hi/lo halves (lo_mask selects lanes that supply
  // the lo halves), value codes as the A operand, zero-point sums as one more tile.
  auto pv = [&](const uint8_t* st, const uint32_t (&ph)[2][2], uint32_t lo_mask) {
#pragma unroll
    for (int hf = 0; hf < 2; ++hf) {
      uint32_t vw[2][CWV];
#pragma unroll
      for (int pi = 0; pi < 2; ++pi)
        lds_chunk<VBITS>(st + St::KB + (8 * hf + 4 * pi + j) * (2 * ROWV) + g * (ROWV / 4), vw[pi]);
      const __half2* vms = reinterpret_cast<const __half2*>(st + St::KB + St::VB) + 16 * hf * NVG;
      __half2 mlo[2 * NVG], mhi[2 * NVG];  // token pairs (2j, 2j+1) and (8+2j, 9+2j)
      lds_vmeta<NVG>(vms + (2 * j) * NVG, mlo);
      lds_vmeta<NVG>(vms + (8 + 2 * j) * NVG, mhi);
      uint32_t bf[NVG][NT][2];
#pragma unroll
      for (int vg = 0; vg < NVG; ++vg) {
        uint32_t za[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint32_t s2 = h2_bits(e ? mhi[2 * vg] : mlo[2 * vg]);  // value scales of the token pair
          const uint32_t whi = hmul2(ph[hf][e], s2);
          if (NT == 1) {
            bf[vg][0][e] = hfma2(ph[hf][e], s2, (whi ^ 0x80008000u) & lo_mask);
          } else {
            bf[vg][0][e] = whi;
            bf[vg][NT - 1][e] = hfma2(ph[hf][e], s2, hneg2(whi));
          }
          za[e] = h2_bits(e ? mhi[2 * vg + 1] : mlo[2 * vg + 1]);  // zero points of the token pair
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(bacc[vg], kOne2, za[0], kOne2, za[1], bf[vg][nt][0], bf[vg][nt][1]);
      }
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const int vg = (mt * NVG) / 8;  // compile-time after unrolling
        const uint32_t a0 = v_pair<VBITS>(vw[0], 2 * mt), a1 = v_pair<VBITS>(vw[0], 2 * mt + 1);
        const uint32_t a2 = v_pair<VBITS>(vw[1], 2 * mt), a3 = v_pair<VBITS>(vw[1], 2 * mt + 1);
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) mma16816(o[mt], a0, a1, a2, a3, bf[vg][nt][0], bf[vg][nt][1]);
      }
    }
  };

  // r <= 4: online softmax of query qj over the lane's tokens 16hf + g and 16hf + 8 + g, then
  // the weights, packed to binary16 and transposed into the B-operand layout of P.V.
  auto softmax_pv_t = [&](int i, const uint8_t* st, const float (&acc)[2][4], float sc, float bi) {
    const int ts = ts0 + i * kTok;
    float s[2][2];  // [hf][e]: token ts + 16hf + 8e + g, log2 units
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int e = 0; e < 2; ++e) s[hf][e] = fmaf(acc[hf][2 * e] + acc[hf][2 * e + 1], sc, bi);
    if constexpr (SYM) {  // score of token t = s_t * (2^24 acc + q_min sum_c q_c), log2 units
      const __half* ksc = reinterpret_cast<const __half*>(st + St::KB + St::VB + St::VM);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float kk = __half2float(ksc[16 * hf + 8 * e + g]);
          s[hf][e] = (kk * p.scale_log2) * fmaf(acc[hf][2 * e] + acc[hf][2 * e + 1], kTwo24, qmin_qsum);
        }
    }
    if constexpr (OUTL) {  // the sparse side list: x_c * q_c of every isolated key entry
      if (SYM || ts < Tq) {  // residual (binary16) keys have no isolated entries
        // lane l takes token l: its entries (channel | binary16 value << 16) against every
        // query row into the warp's table sp_w[token][row] (rows of kMaxGqa + 1 words: no
        // bank conflicts), then every score lane reads its (token, row) term back
        const uint32_t* ent = reinterpret_cast<const uint32_t*>(st + St::KB + St::VB + St::VM + St::KE);
        float* sp_w = reinterpret_cast<float*>(smem + St::SP) + warp * 32 * St::SP_ROW;
        const int ko = p.kout;
        uint32_t en[4];
        if (ko == 4) {
          const uint4 e4 = *reinterpret_cast<const uint4*>(ent + 4 * lane);
          en[0] = e4.x; en[1] = e4.y; en[2] = e4.z; en[3] = e4.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) en[e] = e < ko ? ent[lane * ko + e] : 0u;  // missing: channel 0, value +0
        }
        float xv[4];
        int ch[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xv[e] = __half2float(__ushort_as_half((unsigned short)(en[e] >> 16)));
          ch[e] = (int)(en[e] & (kHeadDim - 1));
        }
        constexpr int kRows = NT == 1 ? 4 : kMaxGqa;
#pragma unroll
        for (int row = 0; row < kRows; ++row)
          if (row < r) {
            float sp = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) sp = fmaf(xv[e], q_s[row][ch[e]], sp);
            sp_w[lane * St::SP_ROW + row] = sp;
          }
        __syncwarp();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int e = 0; e < 2; ++e)
            s[hf][e] = fmaf(sp_w[(16 * hf + 8 * e + g) * St::SP_ROW + qj], p.scale_log2, s[hf][e]);
        __syncwarp();  // the table is rewritten in the next iteration
      }
    }
    if (ts + kTok > t_end) {  // ragged last iteration
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int e = 0; e < 2; ++e)
          if (ts + 16 * hf + 8 * e + g >= t_end) s[hf][e] = -__int_as_float(0x7f800000);
    }
    // lazy rescale as in softmax_pv; the column max gathers the 8 lanes g of query qj
    constexpr float kTau = VBITS == 8 ? 6.0f : (VBITS == 4 ? 2.0f : 0.5f);
    float mx = fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[1][0], s[1][1]));
    if (__any_sync(0xffffffffu, mx > m_run + kTau)) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = ex2(m_run - m_new);  // 0 on the first iteration (m_run = -inf)
      l_run *= alpha;
      // P.V columns 2j, 2j + 1 (and the zero-point tile's) belong to this lane's query
#pragma unroll
      for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int e = 0; e < 4; ++e) o[mt][e] *= alpha;
#pragma unroll
      for (int k = 0; k < NVG; ++k)
#pragma unroll
        for (int e = 0; e < 4; ++e) bacc[k][e] *= alpha;
      m_run = m_new;
    }
    // p rounded once to binary16 (the denominator sums the same values); lane (g, j) holds
    // row g, columns 2j and 2j + 1 of an 8x8 matrix [token][column] whose column n carries
    // query n / 2 — both columns p(token, qj) — and its transpose is the P.V B fragment
    // of column g: tokens (2j, 2j + 1) of query g / 2
    uint32_t ph[2][2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const __half2 h = __float2half2_rn(ex2(s[hf][e] - m_run));
        l_run += __low2float(h);
        ph[hf][e] = movmatrix_t(h2_bits(h));
      }
    pv(st, ph, (g & 1) ? 0xFFFFFFFFu : 0u);  // odd columns carry the lo halves
  };

  // r > 4: online softmax and P.V of iteration i (stage st) from its score accumulators.
  auto softmax_pv = [&](int i, const uint8_t* st, const float (&acc)[2][2][4], float sc, float bi) {
    const int ts = ts0 + i * kTok;
    // scores (log2 units) of tokens ts + 16hf + {2j, 2j+1, 8+2j, 9+2j} for query qi
    float s[2][4];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) s[hf][2 * nt + e] = fmaf(acc[hf][nt][e] + acc[hf][nt][e + 2], sc, bi);
    if constexpr (SYM) {  // score of token t = s_t * (2^24 acc + q_min sum_c q_c), log2 units
      const __half2* ksc = reinterpret_cast<const __half2*>(st + St::KB + St::VB + St::VM);
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          const float2 kk = __half22float2(ksc[8 * hf + 4 * nt + j]);  // tokens 16hf + 8nt + 2j, + 1
          s[hf][2 * nt] = (kk.x * p.scale_log2) * fmaf(acc[hf][nt][0] + acc[hf][nt][2], kTwo24, qmin_qsum);
          s[hf][2 * nt + 1] = (kk.y * p.scale_log2) * fmaf(acc[hf][nt][1] + acc[hf][nt][3], kTwo24, qmin_qsum);
        }
      if constexpr (OUTL) {  // the sparse side list: x_c * q_c of every isolated key entry
        // lane l takes token l: its entries (channel | binary16 value << 16) against every
        // query row into the warp's table sp_w[token][row] (rows of kMaxGqa + 1 words: no
        // bank conflicts), then every score lane reads its (token, row) term back
        const uint32_t* ent = reinterpret_cast<const uint32_t*>(st + St::KB + St::VB + St::VM + St::KE);
        float* sp_w = reinterpret_cast<float*>(smem + St::SP) + warp * 32 * St::SP_ROW;
        const int ko = p.kout;
        uint32_t en[4];
        if (ko == 4) {
          const uint4 e4 = *reinterpret_cast<const uint4*>(ent + 4 * lane);
          en[0] = e4.x; en[1] = e4.y; en[2] = e4.z; en[3] = e4.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) en[e] = e < ko ? ent[lane * ko + e] : 0u;  // missing: channel 0, value +0
        }
        float xv[4];
        int ch[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          xv[e] = __half2float(__ushort_as_half((unsigned short)(en[e] >> 16)));
          ch[e] = (int)(en[e] & (kHeadDim - 1));
        }
        constexpr int kRows = NT == 1 ? 4 : kMaxGqa;
#pragma unroll
        for (int row = 0; row < kRows; ++row)
          if (row < r) {
            float sp = 0.0f;
#pragma unroll
            for (int e = 0; e < 4; ++e) sp = fmaf(xv[e], q_s[row][ch[e]], sp);
            sp_w[lane * St::SP_ROW + row] = sp;
          }
        __syncwarp();
#pragma unroll
        for (int hf = 0; hf < 2; ++hf)
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int tl = 16 * hf + 8 * (k >> 1) + 2 * j + (k & 1);
            s[hf][k] = fmaf(sp_w[tl * St::SP_ROW + qi], p.scale_log2, s[hf][k]);
          }
        __syncwarp();  // the table is rewritten in the next iteration
      }
    }
    if (ts + kTok > t_end) {  // ragged last iteration
#pragma unroll
      for (int hf = 0; hf < 2; ++hf)
#pragma unroll
        for (int k = 0; k < 4; ++k)
          if (ts + 16 * hf + (k >> 1) * 8 + 2 * j + (k & 1) >= t_end) s[hf][k] = -__int_as_float(0x7f800000);
    }
    // Lazy rescale: the running max is only moved when a score exceeds it by more than
    // kTau (log2 units), so p = 2^(s - m_run) <= 2^kTau. kTau keeps every binary16
    // weight p*s finite for any binary16 value group: the largest value scale is
    // 131008 / (2^b - 1) rounded up (514, 8734, 43669 for b = 8, 4, 2). The lane's own
    // scores decide whether any row needs it; only then is the row max gathered.
    constexpr float kTau = VBITS == 8 ? 6.0f : (VBITS == 4 ? 2.0f : 0.5f);
    float mx = fmaxf(fmaxf(fmaxf(s[0][0], s[0][1]), fmaxf(s[0][2], s[0][3])),
                     fmaxf(fmaxf(s[1][0], s[1][1]), fmaxf(s[1][2], s[1][3])));
    if (__any_sync(0xffffffffu, mx > m_run + kTau)) {
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
      const float m_new = fmaxf(m_run, mx);
      const float alpha = ex2(m_run - m_new);  // 0 on the first iteration (m_run = -inf)
      l_run *= alpha;
      // PV column n holds the query of row n: alphas of columns 2j, 2j+1 live in rows 2j, 2j+1
      const float a0 = __shfl_sync(0xffffffffu, alpha, 8 * j);
      const float a1 = __shfl_sync(0xffffffffu, alpha, 8 * j + 4);
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        o[mt][0] *= a0; o[mt][1] *= a1; o[mt][2] *= a0; o[mt][3] *= a1;
      }
#pragma unroll
      for (int k = 0; k < NVG; ++k) {
        bacc[k][0] *= a0; bacc[k][1] *= a1; bacc[k][2] *= a0; bacc[k][3] *= a1;
      }
      m_run = m_new;
    }
    // p = 2^(s - m_run) rounded once to binary16 (token pairs (2j, 2j+1) and (8+2j, 9+2j)
    // of each half). The denominator sums the same rounded values, so the softmax weights
    // are p16 / sum(p16): the rounding perturbs each weight by at most 2^-11 relative and
    // moves an output by at most that times its spread of values. The value weights
    // w = p16 * s are then exact as hi = fl(p16 s), lo = fl(p16 s - hi).
    uint32_t ph[2][2];
#pragma unroll
    for (int hf = 0; hf < 2; ++hf)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const __half2 h = __floats2half2_rn(ex2(s[hf][2 * e] - m_run), ex2(s[hf][2 * e + 1] - m_run));
        const float2 f = __half22float2(h);
        l_run += f.x + f.y;
        ph[hf][e] = h2_bits(h);
      }
    pv(st, ph, 0u);
  };

  int failed_at = -1;
  int sidx = 0;
  uint32_t phase = 0;
  for (int i = 0; i < n_mine; ++i) {
    // every lane takes the same decision (the stage's copies are the whole warp's)
    if (!__all_sync(0xffffffffu, mbar_wait(smem_u32(&bars[warp][sidx]), phase, p.wait_ns))) {
      failed_at = i;
      break;
    }
    const uint8_t* st = wbase + sidx * St::BYTES;
    float sc, bi;
    if constexpr (NT == 1) {
      float acc[2][4];
      qk_t(i, st, acc, sc, bi);
      softmax_pv_t(i, st, acc, sc, bi);
    } else {
      float acc[2][2][4];
      qk(i, st, acc, sc, bi);
      softmax_pv(i, st, acc, sc, bi);
    }
    __syncwarp();  // every lane is done with stage sidx
    if (i + NS < n_mine) issue(i + NS, sidx);
    if (++sidx == NS) {
      sidx = 0;
      phase ^= 1u;
    }
  }

  if (failed_at >= 0) {
    // a stage did not complete in time: flag it (the host reads the word with
    // kvq_decode_error) and drain (bounded) what is still in flight
    if (lane == 0) atomicOr(p.err, KVQ_DECODE_ERR_WAIT_TIMEOUT);
    for (int i = failed_at; i < min(n_mine, failed_at + NS); ++i)
      mbar_wait(smem_u32(&bars[warp][i % NS]), (uint32_t)((i / NS) & 1), kDrainWaitNs);
    asm volatile("cp.async.wait_all;" ::: "memory");  // no copy may land after the CTA exits
  }
  __syncwarp();

  // ---------------- per-warp results -> shared memory (the stage rings are drained)
  __syncthreads();
  float* o_s = reinterpret_cast<float*>(smem);  // [kWarps][kMaxGqa][kHeadDim]
  float* m_s = o_s + kWarps * kMaxGqa * kHeadDim;
  float* l_s = m_s + kWarps * kMaxGqa;
  float* beta_s = l_s + kWarps * kMaxGqa;  // [kWarps][kMaxGqa][NVG]
  if constexpr (NT == 1) {
    // lanes (g, j) hold query j: its denominator over the 8 lanes g, its zero-point sums in
    // columns 2j (hi) and 2j + 1 (lo) of rows 0 (sum w) and 8 (sum zp w), its outputs in
    // columns 2j, 2j + 1 of channel rows g and g + 8 of every m-tile
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 4);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 8);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 16);
    if (g == 0 && j < r) {
      m_s[warp * kMaxGqa + j] = m_run;
      l_s[warp * kMaxGqa + j] = l_run;
#pragma unroll
      for (int k = 0; k < NVG; ++k)
        beta_s[(warp * kMaxGqa + j) * NVG + k] = qmin_v * (bacc[k][0] + bacc[k][1]) - (bacc[k][2] + bacc[k][3]);
    }
    if (j < r) {
#pragma unroll
      for (int mt = 0; mt < 8; ++mt) {
        const float sc0 = 1.0f / v_scale<VBITS>(2 * mt), sc1 = 1.0f / v_scale<VBITS>(2 * mt + 1);
        const int c0 = 16 * mt + g;
        o_s[(warp * kMaxGqa + j) * kHeadDim + c0] = (o[mt][0] + o[mt][1]) * sc0;
        o_s[(warp * kMaxGqa + j) * kHeadDim + c0 + 8] = (o[mt][2] + o[mt][3]) * sc1;
      }
    }
  } else {  // r > 4: row g holds query g; PV columns 2j, 2j + 1 queries 2j, 2j + 1 (hi + lo)
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
    l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    if (j == 0 && g < r) {
      m_s[warp * kMaxGqa + g] = m_run;
      l_s[warp * kMaxGqa + g] = l_run;
    }
    // zero-point terms beta = q_min * sum_t w_t - sum_t zp_t w_t of queries 2j and 2j + 1
#pragma unroll
    for (int k = 0; k < NVG; ++k) {
      if (g == 0) {
        if (2 * j < r) beta_s[(warp * kMaxGqa + 2 * j) * NVG + k] = qmin_v * bacc[k][0] - bacc[k][2];
        if (2 * j + 1 < r) beta_s[(warp * kMaxGqa + 2 * j + 1) * NVG + k] = qmin_v * bacc[k][1] - bacc[k][3];
      }
    }
#pragma unroll
    for (int mt = 0; mt < 8; ++mt) {
      const float sc0 = 1.0f / v_scale<VBITS>(2 * mt), sc1 = 1.0f / v_scale<VBITS>(2 * mt + 1);
      const int i0 = 2 * j, i1 = 2 * j + 1;
      const int c0 = 16 * mt + g, c1 = c0 + 8;
      if (i0 < r) {
        o_s[(warp * kMaxGqa + i0) * kHeadDim + c0] = o[mt][0] * sc0;
        o_s[(warp * kMaxGqa + i0) * kHeadDim + c1] = o[mt][2] * sc1;
      }
      if (i1 < r) {
        o_s[(warp * kMaxGqa + i1) * kHeadDim + c0] = o[mt][1] * sc0;
        o_s[(warp * kMaxGqa + i1) * kHeadDim + c1] = o[mt][3] * sc1;
      }
    }
  }
  __syncthreads();

  // ---------------- CTA merge of the warps; thread = channel (threads 0..127)
  const int c = threadIdx.x;
  const int vgc = ((c & (kHeadDim - 1)) * NVG) / kHeadDim;
  // per-CTA partial (max, denominator, unnormalised output) for the cluster merge
  float* cm_s = reinterpret_cast<float*>(smem + St::EP_CM);  // [kMaxGqa]
  float* cl_s = cm_s + kMaxGqa;                           // [kMaxGqa]
  float* co_s = cl_s + kMaxGqa;                           // [kMaxGqa][kHeadDim]
  for (int i = 0; i < (c < kHeadDim ? r : 0); ++i) {
    float M = -__int_as_float(0x7f800000);
#pragma unroll
    for (int w = 0; w < kWarps; ++w)
      if (((w + 1) * n_it) / kWarps > (w * n_it) / kWarps) M = fmaxf(M, m_s[w * kMaxGqa + i]);
    float L = 0.0f, acc = 0.0f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      if (((w + 1) * n_it) / kWarps == (w * n_it) / kWarps) continue;  // warp had no tokens
      const float wt = ex2(m_s[w * kMaxGqa + i] - M);
      L += wt * l_s[w * kMaxGqa + i];
      acc += wt * fmaf(o_s[(w * kMaxGqa + i) * kHeadDim + c], kTwo24, beta_s[(w * kMaxGqa + i) * NVG + vgc]);
    }
    if (p.cluster == 1) {  // no cluster: this CTA's partial is the split's partial
      if (n_parts == 1) {
        p.out[(qrow0 + i) * kHeadDim + c] = acc / L;
      } else {
        p.ws_o[((qrow0 + i) * p.cap + split) * kHeadDim + c] = acc;
        if (c == 0) p.ws_ml[(qrow0 + i) * p.cap + split] = make_float2(M, L);
      }
      continue;
    }
    co_s[i * kHeadDim + c] = acc;
    if (c == 0) {
      cm_s[i] = M;
      cl_s[i] = L;
    }
  }
  if (p.cluster == 1) {
    // the workspace merge runs with 4-warp CTAs only (the host never plans NW = 8 with parts)
    if constexpr (NW == 4) {
      if (n_parts > 1) merge_if_last(p, n_parts, slice, qrow0, reinterpret_cast<float*>(smem + St::EP_SCRATCH));
    }
    return;
  }
  // ---------------- merge of the splits of one cluster through distributed shared memory.
  // The cluster's CTAs are co-resident and the barriers are hardware cluster barriers.
  // CTA rank R merges channels [R*S, R*S + S) (S = 128 / cluster size) of every query
  // head, reading all partials of the cluster with independent remote loads.
  cg::cluster_group cluster = cg::this_cluster();
  cluster.sync();
  {
    const int cs = p.cluster;  // a power of two <= 16
    const int rank = (int)cluster.block_rank();
    const int S = kHeadDim / cs;
    const int part = split / cs;
    for (int o_idx = threadIdx.x; o_idx < r * S; o_idx += kWarps * 32) {
      const int i = o_idx / S;
      const int cc = rank * S + (o_idx % S);
      float mq[16], lq[16], oq[16];
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        if (q < cs) {
          mq[q] = *cluster.map_shared_rank(cm_s + i, q);
          lq[q] = *cluster.map_shared_rank(cl_s + i, q);
          oq[q] = *cluster.map_shared_rank(co_s + i * kHeadDim + cc, q);
        }
      }
      float M = -__int_as_float(0x7f800000);
#pragma unroll
      for (int q = 0; q < 16; ++q)
        if (q < cs) M = fmaxf(M, mq[q]);
      float L = 0.0f, acc = 0.0f;
#pragma unroll
      for (int q = 0; q < 16; ++q) {
        if (q < cs && mq[q] != -__int_as_float(0x7f800000)) {  // CTAs without tokens weigh 0
          const float wt = ex2(mq[q] - M);
          L += wt * lq[q];
          acc += wt * oq[q];
        }
      }
      if (n_parts == 1) {
        p.out[(qrow0 + i) * kHeadDim + cc] = acc / L;
      } else {
        p.ws_o[((qrow0 + i) * p.cap + part) * kHeadDim + cc] = acc;
        if (rank == 0 && o_idx % S == 0) p.ws_ml[(qrow0 + i) * p.cap + part] = make_float2(M, L);
      }
    }
    if (n_parts > 1) __threadfence();  // slices visible device-wide before the ticket
  }
  cluster.sync();  // the other CTAs keep their shared memory until every rank has read it
  if constexpr (NW == 4) {
    if (n_parts > 1 && cluster.block_rank() == 0)
      merge_if_last(p, n_parts, slice, qrow0, reinterpret_cast<float*>(smem + St::EP_SCRATCH));
  }
}

template <int BITS, int VBITS, int NT, int NVG, int NW, bool SYM, bool OUTL, bool MIXED>
cudaError_t launch_cfg_impl(const DecodeParams& p, cudaStream_t stream) {
  constexpr int smem = Stage<BITS, VBITS, NVG, NW, SYM, OUTL>::SMEM;
  auto* kern = decode_mma_kernel<BITS, VBITS, NT, NVG, NW, SYM, OUTL, MIXED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  if (p.cluster < 1 || p.cluster > 16 || (p.cluster & (p.cluster - 1)) || p.n_split != p.cluster * p.n_parts)
    return cudaErrorInvalidConfiguration;
  if (MIXED && (p.cluster != 1 || p.n_hi < 2 || p.pairs_hi < 1 || p.pairs_hi >= p.B * p.H)) return cudaErrorInvalidConfiguration;
  if (p.cluster > 8) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = MIXED ? dim3((unsigned)(p.pairs_hi * p.n_hi + (p.B * p.H - p.pairs_hi) * (p.n_hi - 1)), 1u, 1u)
                        : dim3((unsigned)p.n_split, (unsigned)p.H, (unsigned)p.B);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)p.cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

template <int BITS, int VBITS, int NT, int NVG, int NW, bool SYM = false, bool OUTL = false>
cudaError_t launch_cfg(const DecodeParams& p, cudaStream_t stream) {
  if constexpr (NW == 4) {
    if (p.mixed) return launch_cfg_impl<BITS, VBITS, NT, NVG, NW, SYM, OUTL, true>(p, stream);
  }
  if (p.mixed) return cudaErrorInvalidConfiguration;  // mixed plans use 4-warp CTAs
  return launch_cfg_impl<BITS, VBITS, NT, NVG, NW, SYM, OUTL, false>(p, stream);
}

template <int BITS, int VBITS, int NT, int NVG, bool SYM = false, bool OUTL = false>
int occupancy_cfg() {
  constexpr int smem = Stage<BITS, VBITS, NVG, 4, SYM, OUTL>::SMEM;
  if (cudaFuncSetAttribute(decode_mma_kernel<BITS, VBITS, NT, NVG, 4, SYM, OUTL>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, decode_mma_kernel<BITS, VBITS, NT, NVG, 4, SYM, OUTL>, 4 * 32,
                                                    smem) !=
      cudaSuccess)
    return 0;
  return n;
}

// Clusters of `cs` CTAs that can be resident at once (0 if such a cluster cannot launch).
template <int BITS, int VBITS, int NT, int NVG, int NW, bool SYM = false, bool OUTL = false>
int max_clusters_cfg(int cs) {
  constexpr int smem = Stage<BITS, VBITS, NVG, NW, SYM, OUTL>::SMEM;
  auto* kern = decode_mma_kernel<BITS, VBITS, NT, NVG, NW, SYM, OUTL>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) return 0;
  if (cs > 8 && cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)cs, 1, 1);
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  return n;
}

template <int BITS, int VBITS, int NW>
int max_clusters_nw(int r, int n_vg, int cs) {
  if (r <= 4) {
    if (n_vg == 1) return max_clusters_cfg<BITS, VBITS, 1, 1, NW>(cs);
    if (n_vg == 2) return max_clusters_cfg<BITS, VBITS, 1, 2, NW>(cs);
    return max_clusters_cfg<BITS, VBITS, 1, 4, NW>(cs);
  }
  if (n_vg == 1) return max_clusters_cfg<BITS, VBITS, 2, 1, NW>(cs);
  if (n_vg == 2) return max_clusters_cfg<BITS, VBITS, 2, 2, NW>(cs);
  return max_clusters_cfg<BITS, VBITS, 2, 4, NW>(cs);
}

template <int BITS, int VBITS>
int max_clusters_bits(int r, int n_vg, int cs, int nw) {
  if (nw == 5) return max_clusters_nw<BITS, VBITS, 5>(r, n_vg, cs);
  return nw == 8 ? max_clusters_nw<BITS, VBITS, 8>(r, n_vg, cs) : max_clusters_nw<BITS, VBITS, 4>(r, n_vg, cs);
}

template <int BITS, int VBITS, int NW>
cudaError_t launch_nw(const DecodeParams& p, cudaStream_t stream) {
  if (p.r <= 4) {
    if (p.n_vg == 1) return launch_cfg<BITS, VBITS, 1, 1, NW>(p, stream);
    if (p.n_vg == 2) return launch_cfg<BITS, VBITS, 1, 2, NW>(p, stream);
    return launch_cfg<BITS, VBITS, 1, 4, NW>(p, stream);
  }
  if (p.n_vg == 1) return launch_cfg<BITS, VBITS, 2, 1, NW>(p, stream);
  if (p.n_vg == 2) return launch_cfg<BITS, VBITS, 2, 2, NW>(p, stream);
  return launch_cfg<BITS, VBITS, 2, 4, NW>(p, stream);
}

template <int BITS, int VBITS>
cudaError_t launch_bits(const DecodeParams& p, cudaStream_t stream) {
  if (p.warps == 8 || p.warps == 5) {
    if (p.n_parts != 1) return cudaErrorInvalidConfiguration;  // 5- and 8-warp CTAs merge in clusters only
    return p.warps == 8 ? launch_nw<BITS, VBITS, 8>(p, stream) : launch_nw<BITS, VBITS, 5>(p, stream);
  }
  return launch_nw<BITS, VBITS, 4>(p, stream);
}

template <int BITS, int VBITS>
int occupancy_bits(int r, int n_vg) {
  if (r <= 4) {
    if (n_vg == 1) return occupancy_cfg<BITS, VBITS, 1, 1>();
    if (n_vg == 2) return occupancy_cfg<BITS, VBITS, 1, 2>();
    return occupancy_cfg<BITS, VBITS, 1, 4>();
  }
  if (n_vg == 1) return occupancy_cfg<BITS, VBITS, 2, 1>();
  if (n_vg == 2) return occupancy_cfg<BITS, VBITS, 2, 2>();
  return occupancy_cfg<BITS, VBITS, 2, 4>();
}

}  // namespace mma
}  // namespace kvq
