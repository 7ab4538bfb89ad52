// kvq_oracle.cpp — TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU statement of what the quantized KV cache and
// its decode attention compute. Only the test suite, the smoke check and the CPU
// baseline leg of the benchmark load this file's library; the product path never
// does. It shares no code, header, table or constant with the CUDA library.
//
// Build: g++ -std=c++17 -O2 -ffp-contract=off -fno-fast-math -shared -fPIC
// (no FMA contraction: every float operation below is one IEEE-754 binary32
// operation rounded to nearest-even, in the order written).
//
// Sources (web pages; titles and sections):
//   [A] "KV Cache Quantization — 8-bit and 4-bit"
//       § The bytes-per-token formula; § A worked memory example;
//       § Integer quantization in one screen; § Granularity: per-tensor, per-token,
//       per-channel; § The outlier problem: keys have outlier channels;
//       § Why keys and values want different treatment.
//   [B] "Sub-8-Bit KV Cache Quantization Is Not a Free Lever for an RDNA4 Agent Swarm"
//       § The cache is two distributions, not one (keys per channel, values per token);
//       § What the low-bit numbers actually cost (full-precision residual of recent tokens).
//   [C] "KV Cache Quantization Benchmarked: 8-bit Is Nearly Lossless, How Much Does
//       4-bit Cost?" § KV Cache Quantization: 8-bit Is Essentially Free (64k-context
//       bytes with one 16-bit scale per 32-element block).
//
// Readings where the pages leave a step open (each one is listed with its reason in
// the design notes):
//   round()          -> round half to even, in binary32.
//   stored scale     -> binary16, rounded toward +infinity from the binary32 quotient,
//                       and the quantizer divides by that stored value.
//   zero point       -> binary16 (an integer, exact there), and the quantizer adds
//                       that stored value; a narrow group far from zero, whose zero
//                       point would exceed the binary16 integers (2048), gets the
//                       wider scale max|x| / (2048 - 2^bits) instead.
//   q = clamp(round(x/scale) + zero_point, q_min, q_max), codes kept as u = q - q_min.
//   int2 range       -> [-2, 1].
//   degenerate group -> if x_max == x_min widen the range to include 0; if it is still
//                       empty (all zeros) the scale is 1.
//   residual window  -> keys only; it holds the T mod R_eff newest tokens (R_eff = R,
//                       or G when R = 0) and is quantized R_eff tokens at a time.
//   symmetric scheme -> scale = max|x| / q_max rounded up to binary16, zero point 0,
//                       one scale per token for keys and values, no residual window.
//   outlier isolation-> per key row (either scheme): the k channels farthest from the
//                       row's lower median in |x - median| (binary32), ties to the lower
//                       channel, kept as (channel, binary16 value) and zeroed in the
//                       dense row that is then quantized (per token in the symmetric
//                       scheme; with per-channel keys, when the row's group is formed).
//
// Parity pins: see tests/test_oracle_pins.py. The packed byte layout and the
// residual/flush bookkeeping are this project's own definitions (the pages fix
// neither). The layout functions are pinned against bytes derived by hand from the
// layout's written rules (tests/golden/layout_bytes.json); the flush bookkeeping by
// chunking invariance and the residual-window tests.

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <vector>

extern "C" {

// ---------------------------------------------------------------------------
// binary16 <-> binary32, written from the IEEE-754 bit layouts.
// binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
// ---------------------------------------------------------------------------

float orc_f32_from_f16(uint16_t h) {
  uint32_t sign = (uint32_t)(h >> 15) & 1u;
  uint32_t e = (uint32_t)(h >> 10) & 0x1Fu;
  uint32_t f = (uint32_t)h & 0x3FFu;
  double mag;
  if (e == 0x1F) {
    mag = f ? NAN : INFINITY;
  } else if (e == 0) {
    mag = std::ldexp((double)f, -24);  // subnormal: f * 2^-24
  } else {
    mag = std::ldexp((double)(1024u + f), (int)e - 25);  // (1024+f) * 2^(e-15-10)
  }
  double v = sign ? -mag : mag;
  return (float)v;  // exact: every binary16 value is a binary32 value
}

// Round a finite binary32 value to binary16. mode 0 = nearest, ties to even;
// mode 1 = toward +infinity. Overflow follows IEEE: nearest-even gives +-inf at
// |x| >= 65520; toward +inf gives +inf above 65504 and -65504 for x < -65504.
static uint16_t f16_round(float x, int mode) {
  if (std::isnan(x)) return 0x7E00;
  uint16_t sign = std::signbit(x) ? 0x8000 : 0;
  if (std::isinf(x)) {
    if (!sign) return 0x7C00;
    return mode == 1 ? (uint16_t)0xFBFF : (uint16_t)0xFC00;
  }
  double a = std::fabs((double)x);
  if (a == 0.0) return sign;
  // The binary16 quantum at |x|: 2^(max(floor(log2 a), -14) - 10).
  int ex;
  std::frexp(a, &ex);  // a = m * 2^ex, m in [0.5, 1)  =>  floor(log2 a) = ex - 1
  int e2 = ex - 1;
  if (e2 < -14) e2 = -14;
  double n = std::ldexp(a, 10 - e2);  // exact: a has 24 significant bits
  double fl = std::floor(n);
  double rem = n - fl;  // exact
  double k;             // rounded magnitude in quanta
  if (mode == 0) {
    if (rem > 0.5) k = fl + 1;
    else if (rem < 0.5) k = fl;
    else k = (std::fmod(fl, 2.0) == 0.0) ? fl : fl + 1;
  } else {
    // toward +inf: magnitude rounds up for positive x, down (truncates) for negative x
    if (!sign) k = (rem > 0) ? fl + 1 : fl;
    else k = fl;
  }
  // k is in [0, 2048]; 2048 moves to the next binade.
  double val = std::ldexp(k, e2 - 10);
  if (val > 65504.0) {
    if (mode == 0) return (uint16_t)(sign | 0x7C00);
    return sign ? (uint16_t)0xFBFF : (uint16_t)0x7C00;
  }
  if (val == 0.0) return sign;
  int vex;
  std::frexp(val, &vex);
  int ve = vex - 1;  // floor(log2 val)
  if (ve < -14) {
    // subnormal: val = f * 2^-24
    uint32_t f = (uint32_t)std::ldexp(val, 24);
    return (uint16_t)(sign | f);
  }
  uint32_t mant = (uint32_t)std::ldexp(val, 10 - ve);  // in [1024, 2047]
  uint32_t ebits = (uint32_t)(ve + 15);
  return (uint16_t)(sign | (ebits << 10) | (mant - 1024u));
}

uint16_t orc_f16_from_f32_rne(float x) { return f16_round(x, 0); }
uint16_t orc_f16_from_f32_ru(float x) { return f16_round(x, 1); }

// Round half to even of a binary32 value, to an integral binary32 value.
static float rne_integral(float t) {
  float fl = std::floor(t);
  float diff = t - fl;  // exact (Sterbenz-range / integral part removed)
  if (diff > 0.5f) return fl + 1.0f;
  if (diff < 0.5f) return fl;
  return (std::fmod(fl, 2.0f) == 0.0f) ? fl : fl + 1.0f;
}

// ---------------------------------------------------------------------------
// Affine quantizer, [A] § Integer quantization in one screen:
//   scale      = (x_max - x_min) / (q_max - q_min)
//   zero_point = q_min - round(x_min / scale)
//   q          = round(x / scale) + zero_point      (clamped to [q_min, q_max])
//   x_hat      = scale * (q - zero_point)
// with int8 range [-128, 127], int4 [-8, 7] (and int2 read as [-2, 1]).
// ---------------------------------------------------------------------------

static int qmin_of(int bits) { return -(1 << (bits - 1)); }
static int qmax_of(int bits) { return (1 << (bits - 1)) - 1; }

int orc_qmin(int bits) { return qmin_of(bits); }
int orc_qmax(int bits) { return qmax_of(bits); }

// Group parameters for n binary16 values x[0], x[stride], ...
// Returns 0 on success, -1 on a bad argument.
int orc_quant_params(const uint16_t* x, int64_t n, int64_t stride, int bits, uint16_t* scale_h, uint16_t* zp_h) {
  if (n <= 0 || !(bits == 2 || bits == 4 || bits == 8)) return -1;
  float xmin = orc_f32_from_f16(x[0]);
  float xmax = xmin;
  for (int64_t i = 1; i < n; ++i) {
    float v = orc_f32_from_f16(x[i * stride]);
    if (v < xmin) xmin = v;
    if (v > xmax) xmax = v;
  }
  if (xmax == xmin) {  // degenerate group: include 0 in the range
    if (xmin > 0.0f) xmin = 0.0f;
    if (xmax < 0.0f) xmax = 0.0f;
  }
  const int qmin = qmin_of(bits), qmax = qmax_of(bits);
  uint16_t s_h;
  if (xmax == xmin) {
    s_h = 0x3C00;  // all zeros: scale 1
  } else {
    float range = xmax - xmin;                  // binary32, nearest-even
    float s32 = range / (float)(qmax - qmin);   // binary32, nearest-even
    // The zero point is stored in binary16, which holds every integer only up to 2048.
    // A narrow group far from zero would need a larger one, so its scale is widened to
    // max|x| / (2048 - 2^bits): then |x / scale| <= 2048 - 2^bits for every x of the
    // group, |zero_point| <= 2048 - 2^(bits-1) is stored exactly, and the half-step
    // bound |x - x_hat| <= scale/2 holds with the stored (wider) scale.
    float amax = std::fabs(xmin) > std::fabs(xmax) ? std::fabs(xmin) : std::fabs(xmax);
    float s_far = amax / (float)(2048 - (1 << bits));  // binary32, nearest-even
    if (s_far > s32) s32 = s_far;
    s_h = orc_f16_from_f32_ru(s32);             // stored scale, rounded up
  }
  float s = orc_f32_from_f16(s_h);
  float t = xmin / s;
  float zp = (float)qmin - rne_integral(t);     // an integer of magnitude <= 2048
  *scale_h = s_h;
  *zp_h = orc_f16_from_f32_rne(zp);
  return 0;
}

// u = clamp(round(x / scale) + zero_point, q_min, q_max) - q_min for n values.
int orc_quantize_values(const uint16_t* x, int64_t n, int64_t stride, int bits, uint16_t scale_h, uint16_t zp_h,
                        uint8_t* u_out) {
  if (n < 0 || !(bits == 2 || bits == 4 || bits == 8)) return -1;
  const float s = orc_f32_from_f16(scale_h);
  const float zp = orc_f32_from_f16(zp_h);
  const float qmin = (float)qmin_of(bits), qmax = (float)qmax_of(bits);
  for (int64_t i = 0; i < n; ++i) {
    float v = orc_f32_from_f16(x[i * stride]);
    float q = rne_integral(v / s) + zp;
    if (q < qmin) q = qmin;
    if (q > qmax) q = qmax;
    u_out[i] = (uint8_t)(int)(q - qmin);
  }
  return 0;
}

// x_hat = scale * (q - zero_point), one binary32 product.
float orc_dequantize_value(int u, int bits, uint16_t scale_h, uint16_t zp_h) {
  float q = (float)(u + qmin_of(bits));
  float diff = q - orc_f32_from_f16(zp_h);  // exact: integers below 2^17
  return orc_f32_from_f16(scale_h) * diff;
}

// ---------------------------------------------------------------------------
// Bytes accounting, [A] § The bytes-per-token formula:
//   bytes = 2 * L * n_kv * d_head * S * bytes_per_elem
// bytes_per_elem is given here as bits/8 so that int4 (0.5 B) is exact, plus a
// metadata term: meta_bytes per group of group_elems elements (0 = none).
// ---------------------------------------------------------------------------

double orc_kv_bytes(int64_t L, int64_t n_kv, int64_t d_head, int64_t S, double bits_per_elem, double meta_bytes,
                    double group_elems) {
  double elems = 2.0 * (double)L * (double)n_kv * (double)d_head * (double)S;
  double per = bits_per_elem / 8.0;
  if (group_elems > 0) per += meta_bytes / group_elems;
  return elems * per;
}

// ---------------------------------------------------------------------------
// Packed layout (this project's definition; pinned by hand-derived bytes).
//   Key row (one token, d channels): channel c occupies bits [c*b, c*b + b) of the
//   row, little-endian bytes, low bits first.
//   Value rows: channel c is stored at position
//     pos(c) = (d/8) * (c % 8) + 2 * (c / 16) + (c / 8) % 2
//   of the token's row (bits [pos*b, pos*b + b)), and the rows of tokens 2p and
//   2p+1 are interleaved in 16-bit units: 32-bit word k of pair row p holds 16-bit
//   unit k of token 2p in its low half and unit k of token 2p+1 in its high half.
//   Key metadata entries are (scale, zero_point) binary16 pairs.
//   Value metadata is stored per token pair: for tokens 2p and 2p+1 and value group j,
//   the record at [p][j] holds four binary16 values, {scale of 2p, scale of 2p+1,
//   zero point of 2p, zero point of 2p+1}.
// ---------------------------------------------------------------------------

static void put_bits(uint8_t* row, int64_t pos, int bits, uint32_t u) {
  int64_t bit = pos * bits;
  for (int i = 0; i < bits; ++i) {
    int64_t b = bit + i;
    if ((u >> i) & 1u) row[b >> 3] = (uint8_t)(row[b >> 3] | (1u << (b & 7)));
    else row[b >> 3] = (uint8_t)(row[b >> 3] & ~(1u << (b & 7)));
  }
}

static uint32_t get_bits(const uint8_t* row, int64_t pos, int bits) {
  int64_t bit = pos * bits;
  uint32_t u = 0;
  for (int i = 0; i < bits; ++i) {
    int64_t b = bit + i;
    u |= (uint32_t)((row[b >> 3] >> (b & 7)) & 1u) << i;
  }
  return u;
}

int64_t orc_v_pos(int d, int c) { return (int64_t)(d / 8) * (c % 8) + 2 * (c / 16) + (c / 8) % 2; }

// Index (in binary16 units) of token t's scale (part 0) or zero point (part 1) of value
// group j, with ng groups per token, in the pair records described above.
int64_t orc_v_meta_index(int64_t t, int ng, int j, int part) { return ((t / 2) * ng + j) * 4 + 2 * part + t % 2; }

// Key row: u[d] codes -> row bytes (d*b/8).
void orc_pack_k_row(const uint8_t* u, int d, int bits, uint8_t* row) {
  std::memset(row, 0, (size_t)d * bits / 8);
  for (int c = 0; c < d; ++c) put_bits(row, c, bits, u[c]);
}

void orc_unpack_k_row(const uint8_t* row, int d, int bits, uint8_t* u) {
  for (int c = 0; c < d; ++c) u[c] = (uint8_t)get_bits(row, c, bits);
}

// Value token t (codes u[d]) written into its half of pair row (t/2) of `pairs`.
void orc_pack_v_token(const uint8_t* u, int d, int bits, int64_t t, uint8_t* pairs) {
  const int64_t row_bytes = (int64_t)d * bits / 8;
  std::vector<uint8_t> row((size_t)row_bytes, 0);
  for (int c = 0; c < d; ++c) put_bits(row.data(), orc_v_pos(d, c), bits, u[c]);
  uint8_t* pr = pairs + (t / 2) * 2 * row_bytes;
  const int half = (int)(t % 2);
  for (int64_t k = 0; k < row_bytes / 2; ++k) {
    pr[4 * k + 2 * half + 0] = row[2 * k + 0];
    pr[4 * k + 2 * half + 1] = row[2 * k + 1];
  }
}

void orc_unpack_v_token(const uint8_t* pairs, int d, int bits, int64_t t, uint8_t* u) {
  const int64_t row_bytes = (int64_t)d * bits / 8;
  std::vector<uint8_t> row((size_t)row_bytes, 0);
  const uint8_t* pr = pairs + (t / 2) * 2 * row_bytes;
  const int half = (int)(t % 2);
  for (int64_t k = 0; k < row_bytes / 2; ++k) {
    row[2 * k + 0] = pr[4 * k + 2 * half + 0];
    row[2 * k + 1] = pr[4 * k + 2 * half + 1];
  }
  for (int c = 0; c < d; ++c) u[c] = (uint8_t)get_bits(row.data(), orc_v_pos(d, c), bits);
}

// ---------------------------------------------------------------------------
// Cache state of one (batch row, kv head) after T tokens, [B] § The cache is two
// distributions, not one, and § What the low-bit numbers actually cost:
//   keys   : per channel, over groups of G consecutive tokens; the newest
//            T mod R_eff tokens stay binary16 in the residual window (slot t mod R_eff);
//   values : per token, over groups of Gv consecutive channels.
// Keys use `bits`-bit codes (b), values `v_bits`-bit codes (b_v; equal to b unless a
// mixed-width cache is asked for, "KV Cache Quantization — 8-bit and 4-bit", § Why keys
// and values want different treatment).
// Inputs k_hist, v_hist: [T][d] binary16. Outputs in the packed layout above:
//   k_codes [floor(T/R_eff)*R_eff][d*b/8], k_meta [groups][d][2], k_resid [R_eff][d],
//   v_codes [ceil(T/2)][2*d*b_v/8], v_meta [ceil(T/2)][d/Gv][4]; with k_out > 0 isolated key entries
//   per quantized row, k_sparse [Tq][k_out][2] (see below).
// Output buffers must be zero-initialised by the caller. Optional k_u [Tq][d] and
// v_u [T][d] receive the unpacked codes. Returns Tq (quantized key tokens) or -1.
// ---------------------------------------------------------------------------

int orc_split_outliers(const uint16_t* x, int n, int k, uint16_t* idx_out, uint16_t* val_out, uint16_t* dense_out);

int64_t orc_cache_state(int d, int bits, int v_bits, int G, int Gv, int R, int64_t T, int k_out,
                        const uint16_t* k_hist, const uint16_t* v_hist, uint8_t* k_codes, uint16_t* k_meta,
                        uint16_t* k_sparse, uint16_t* k_resid, uint8_t* v_codes, uint16_t* v_meta, uint8_t* k_u,
                        uint8_t* v_u) {
  if (d <= 0 || d % 16 || G <= 0 || Gv <= 0 || d % Gv || R < 0 || (R > 0 && R % G) || T < 0) return -1;
  if (k_out < 0 || k_out > d) return -1;
  if (!(bits == 2 || bits == 4 || bits == 8)) return -1;
  if (!(v_bits == 2 || v_bits == 4 || v_bits == 8)) return -1;
  const int64_t R_eff = R > 0 ? R : G;
  const int64_t Tq = (T / R_eff) * R_eff;
  const int64_t rowK = (int64_t)d * bits / 8;
  std::vector<uint8_t> u((size_t)d);
  std::vector<uint8_t> col((size_t)G);
  // Dense-and-sparse keys (k_out > 0): every key row that is quantized first gives up its
  // k_out entries farthest from its lower median (orc_split_outliers), kept as
  // (channel, binary16 value) in k_sparse [Tq][k_out][2]; the per-channel groups are
  // then formed over the dense rows. Residual rows stay whole (they are binary16 already).
  std::vector<uint16_t> dense((size_t)(Tq > 0 ? Tq : 1) * d);
  std::vector<uint16_t> idx((size_t)k_out + 1), val((size_t)k_out + 1);
  for (int64_t t = 0; t < Tq; ++t) {
    if (k_out > 0) {
      orc_split_outliers(k_hist + t * d, d, k_out, idx.data(), val.data(), dense.data() + t * d);
      for (int r = 0; r < k_out; ++r) {
        k_sparse[(t * k_out + r) * 2 + 0] = idx[(size_t)r];
        k_sparse[(t * k_out + r) * 2 + 1] = val[(size_t)r];
      }
    } else {
      std::memcpy(dense.data() + t * d, k_hist + t * d, sizeof(uint16_t) * (size_t)d);
    }
  }
  // keys: per channel, per group of G tokens
  for (int64_t g = 0; g < Tq / G; ++g) {
    for (int c = 0; c < d; ++c) {
      const uint16_t* x = dense.data() + (g * G) * d + c;
      uint16_t s_h, z_h;
      orc_quant_params(x, G, d, bits, &s_h, &z_h);
      orc_quantize_values(x, G, d, bits, s_h, z_h, col.data());
      k_meta[(g * d + c) * 2 + 0] = s_h;
      k_meta[(g * d + c) * 2 + 1] = z_h;
      for (int i = 0; i < G; ++i) {
        int64_t t = g * G + i;
        put_bits(k_codes + t * rowK, c, bits, col[(size_t)i]);
        if (k_u) k_u[t * d + c] = col[(size_t)i];
      }
    }
  }
  // residual window: binary16 copies of tokens [Tq, T)
  for (int64_t t = Tq; t < T; ++t) {
    std::memcpy(k_resid + (t % R_eff) * d, k_hist + t * d, sizeof(uint16_t) * (size_t)d);
  }
  // values: per token, per group of Gv channels
  const int ng = d / Gv;
  for (int64_t t = 0; t < T; ++t) {
    for (int j = 0; j < ng; ++j) {
      const uint16_t* x = v_hist + t * d + (int64_t)j * Gv;
      uint16_t s_h, z_h;
      orc_quant_params(x, Gv, 1, v_bits, &s_h, &z_h);
      orc_quantize_values(x, Gv, 1, v_bits, s_h, z_h, u.data() + (size_t)j * Gv);
      v_meta[orc_v_meta_index(t, ng, j, 0)] = s_h;
      v_meta[orc_v_meta_index(t, ng, j, 1)] = z_h;
    }
    orc_pack_v_token(u.data(), d, v_bits, t, v_codes);
    if (v_u) std::memcpy(v_u + t * d, u.data(), (size_t)d);
  }
  return Tq;
}

// Dequantized keys and values of one (batch row, kv head) from a packed state:
// k_out, v_out [T][d] binary32. Quantized keys and all values use
// x_hat = scale * (q - zero_point); residual keys are the binary16 values.
int orc_dequantize_state(int d, int bits, int v_bits, int G, int Gv, int R, int64_t T, int k_out_n,
                         const uint8_t* k_codes, const uint16_t* k_meta, const uint16_t* k_sparse,
                         const uint16_t* k_resid, const uint8_t* v_codes, const uint16_t* v_meta, float* k_out,
                         float* v_out) {
  if (d <= 0 || d % 16 || G <= 0 || Gv <= 0 || d % Gv || R < 0 || (R > 0 && R % G) || T < 0) return -1;
  const int64_t R_eff = R > 0 ? R : G;
  const int64_t Tq = (T / R_eff) * R_eff;
  const int64_t rowK = (int64_t)d * bits / 8;
  std::vector<uint8_t> u((size_t)d);
  for (int64_t t = 0; t < T; ++t) {
    if (t < Tq) {
      int64_t g = t / G;
      orc_unpack_k_row(k_codes + t * rowK, d, bits, u.data());
      for (int c = 0; c < d; ++c)
        k_out[t * d + c] = orc_dequantize_value(u[(size_t)c], bits, k_meta[(g * d + c) * 2], k_meta[(g * d + c) * 2 + 1]);
      for (int r = 0; r < k_out_n; ++r)  // isolated entries: the dense x_hat there is 0 + its own error
        k_out[t * d + k_sparse[(t * k_out_n + r) * 2]] += orc_f32_from_f16(k_sparse[(t * k_out_n + r) * 2 + 1]);
    } else {
      for (int c = 0; c < d; ++c) k_out[t * d + c] = orc_f32_from_f16(k_resid[(t % R_eff) * d + c]);
    }
    const int ng = d / Gv;
    orc_unpack_v_token(v_codes, d, v_bits, t, u.data());
    for (int c = 0; c < d; ++c) {
      int j = c / Gv;
      v_out[t * d + c] = orc_dequantize_value(u[(size_t)c], v_bits, v_meta[orc_v_meta_index(t, ng, j, 0)],
                                              v_meta[orc_v_meta_index(t, ng, j, 1)]);
    }
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Symmetric quantizer, [A] § Symmetric vs asymmetric: the zero point is forced to 0
// and the integer range is centred on real zero, x_hat = scale * q. Readings:
//   scale  = max|x| / q_max (q_max = 2^(b-1) - 1), stored as binary16 rounded toward
//            +infinity (so |x| / scale <= q_max), and the quantizer divides by it;
//            an all-zero vector gets scale 1;
//   q      = clamp(round(x / scale), q_min, q_max), kept as u = q - q_min.
// ---------------------------------------------------------------------------

int orc_sym_params(const uint16_t* x, int64_t n, int64_t stride, int bits, uint16_t* scale_h) {
  if (n <= 0 || !(bits == 2 || bits == 4 || bits == 8)) return -1;
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float v = std::fabs(orc_f32_from_f16(x[i * stride]));
    if (v > amax) amax = v;
  }
  if (amax == 0.0f) {
    *scale_h = 0x3C00;  // all zeros: scale 1
  } else {
    float s32 = amax / (float)qmax_of(bits);  // binary32, nearest-even
    *scale_h = orc_f16_from_f32_ru(s32);
  }
  return 0;
}

int orc_sym_quantize(const uint16_t* x, int64_t n, int64_t stride, int bits, uint16_t scale_h, uint8_t* u_out) {
  if (n < 0 || !(bits == 2 || bits == 4 || bits == 8)) return -1;
  const float s = orc_f32_from_f16(scale_h);
  const float qmin = (float)qmin_of(bits), qmax = (float)qmax_of(bits);
  for (int64_t i = 0; i < n; ++i) {
    float q = rne_integral(orc_f32_from_f16(x[i * stride]) / s);
    if (q < qmin) q = qmin;
    if (q > qmax) q = qmax;
    u_out[i] = (uint8_t)(int)(q - qmin);
  }
  return 0;
}

// x_hat = scale * q, one binary32 product.
float orc_sym_dequantize_value(int u, int bits, uint16_t scale_h) {
  return orc_f32_from_f16(scale_h) * (float)(u + qmin_of(bits));
}

// Dense-and-sparse split of one vector of n binary16 values ("Sub-8-Bit KV Cache
// Quantization Is Not a Free Lever for an RDNA4 Agent Swarm", § What the low-bit numbers
// actually cost: per-vector dense-and-sparse quantization pulls the outliers out and
// stores them separately; § The RDNA4 kernel angle: a sparse side channel read alongside
// the dense one). The pages fix neither the rule nor k; here: the k entries farthest from
// the vector's lower median (the ((n-1)/2)-th smallest value, counting from 0) in
// binary32 |x - median|, taken in order of decreasing distance, ties to the lower index.
// They go to idx_out/val_out (channel, binary16 value) and become +0 in dense_out.
int orc_split_outliers(const uint16_t* x, int n, int k, uint16_t* idx_out, uint16_t* val_out, uint16_t* dense_out) {
  if (n <= 0 || k < 0 || k > n) return -1;
  std::vector<float> v((size_t)n), sorted((size_t)n), dist((size_t)n);
  for (int c = 0; c < n; ++c) v[(size_t)c] = sorted[(size_t)c] = orc_f32_from_f16(x[c]);
  std::sort(sorted.begin(), sorted.end());
  const float med = sorted[(size_t)((n - 1) / 2)];
  for (int c = 0; c < n; ++c) dist[(size_t)c] = std::fabs(v[(size_t)c] - med);
  std::vector<char> taken((size_t)n, 0);
  for (int c = 0; c < n; ++c) dense_out[c] = x[c];
  for (int r = 0; r < k; ++r) {
    int best = -1;
    for (int c = 0; c < n; ++c)
      if (!taken[(size_t)c] && (best < 0 || dist[(size_t)c] > dist[(size_t)best])) best = c;
    taken[(size_t)best] = 1;
    idx_out[r] = (uint16_t)best;
    val_out[r] = x[best];
    dense_out[best] = 0;  // binary16 +0
  }
  return 0;
}

// Symmetric per-token int8 cache of one (batch row, kv head) after T tokens ("Sub-8-Bit
// KV Cache Quantization Is Not a Free Lever for an RDNA4 Agent Swarm", § The RDNA4
// kernel angle: one scale per token; [A] § Symmetric vs asymmetric): keys and values
// are each quantized per token over all d channels with the symmetric quantizer; there
// is no residual window. Layout: k_codes [T][d] (key rows as above), k_scale [T]
// binary16, v_codes pair rows as above, v_meta [ceil(T/2)][1][4] pair records with
// zero points +0. Optional k_u,
// v_u [T][d] receive the unpacked codes. Returns 0, or -1 on a bad argument.
// With k_out > 0 outliers per key row (see orc_split_outliers), the dense row is what
// is quantized and k_sparse [T][k_out][2] receives the (channel, binary16 value) pairs.
int orc_cache_state_sym(int d, int64_t T, int k_out, const uint16_t* k_hist, const uint16_t* v_hist, uint8_t* k_codes,
                        uint16_t* k_scale, uint16_t* k_sparse, uint8_t* v_codes, uint16_t* v_meta, uint8_t* k_u,
                        uint8_t* v_u) {
  if (d <= 0 || d % 16 || T < 0 || k_out < 0 || k_out > d) return -1;
  const int bits = 8;
  std::vector<uint8_t> u((size_t)d);
  std::vector<uint16_t> dense((size_t)d), idx((size_t)k_out + 1), val((size_t)k_out + 1);
  for (int64_t t = 0; t < T; ++t) {
    uint16_t s_h;
    const uint16_t* krow = k_hist + t * d;
    if (k_out > 0) {
      orc_split_outliers(krow, d, k_out, idx.data(), val.data(), dense.data());
      for (int r = 0; r < k_out; ++r) {
        k_sparse[(t * k_out + r) * 2 + 0] = idx[(size_t)r];
        k_sparse[(t * k_out + r) * 2 + 1] = val[(size_t)r];
      }
      krow = dense.data();
    }
    orc_sym_params(krow, d, 1, bits, &s_h);
    orc_sym_quantize(krow, d, 1, bits, s_h, u.data());
    k_scale[t] = s_h;
    orc_pack_k_row(u.data(), d, bits, k_codes + t * d);
    if (k_u) std::memcpy(k_u + t * d, u.data(), (size_t)d);
    orc_sym_params(v_hist + t * d, d, 1, bits, &s_h);
    orc_sym_quantize(v_hist + t * d, d, 1, bits, s_h, u.data());
    v_meta[orc_v_meta_index(t, 1, 0, 0)] = s_h;
    v_meta[orc_v_meta_index(t, 1, 0, 1)] = 0;  // binary16 +0
    orc_pack_v_token(u.data(), d, bits, t, v_codes);
    if (v_u) std::memcpy(v_u + t * d, u.data(), (size_t)d);
  }
  return 0;
}

// Dequantized keys and values of a symmetric per-token state: k_out, v_out [T][d]. With
// k_out_n > 0 outliers per key row the stored binary16 values replace the dense x_hat
// (which is 0 there) at their channels.
int orc_dequantize_state_sym(int d, int64_t T, int k_out_n, const uint8_t* k_codes, const uint16_t* k_scale,
                             const uint16_t* k_sparse, const uint8_t* v_codes, const uint16_t* v_meta, float* k_out,
                             float* v_out) {
  if (d <= 0 || d % 16 || T < 0 || k_out_n < 0) return -1;
  const int bits = 8;
  std::vector<uint8_t> u((size_t)d);
  for (int64_t t = 0; t < T; ++t) {
    orc_unpack_k_row(k_codes + t * d, d, bits, u.data());
    for (int c = 0; c < d; ++c) k_out[t * d + c] = orc_sym_dequantize_value(u[(size_t)c], bits, k_scale[t]);
    for (int r = 0; r < k_out_n; ++r)
      k_out[t * d + k_sparse[(t * k_out_n + r) * 2]] += orc_f32_from_f16(k_sparse[(t * k_out_n + r) * 2 + 1]);
    orc_unpack_v_token(v_codes, d, bits, t, u.data());
    for (int c = 0; c < d; ++c)
      v_out[t * d + c] = orc_sym_dequantize_value(u[(size_t)c], bits, v_meta[orc_v_meta_index(t, 1, 0, 0)]);
  }
  return 0;
}

// ---------------------------------------------------------------------------
// Decode attention for one (batch row, kv head) and its r query heads, exact
// softmax in binary64 over the dequantized binary32 keys and values:
//   z_t = softmax_scale * sum_c q_c * k_hat[t][c]
//   p_t = exp(z_t - max z) / sum exp(z - max z)
//   o_c = sum_t p_t * v_hat[t][c]
// q [r][d] binary16, k_hat/v_hat [T][d], out [r][d] binary32.
// ---------------------------------------------------------------------------

int orc_attention(int d, int r, int64_t T, const uint16_t* q, const float* k_hat, const float* v_hat,
                  float softmax_scale, float* out) {
  if (T <= 0 || d <= 0 || r <= 0) return -1;
  std::vector<double> z((size_t)T);
  for (int i = 0; i < r; ++i) {
    double zmax = -INFINITY;
    for (int64_t t = 0; t < T; ++t) {
      double acc = 0.0;
      for (int c = 0; c < d; ++c) acc += (double)orc_f32_from_f16(q[i * d + c]) * (double)k_hat[t * d + c];
      z[(size_t)t] = (double)softmax_scale * acc;
      if (z[(size_t)t] > zmax) zmax = z[(size_t)t];
    }
    double denom = 0.0;
    for (int64_t t = 0; t < T; ++t) {
      z[(size_t)t] = std::exp(z[(size_t)t] - zmax);
      denom += z[(size_t)t];
    }
    for (int c = 0; c < d; ++c) {
      double acc = 0.0;
      for (int64_t t = 0; t < T; ++t) acc += z[(size_t)t] * (double)v_hat[t * d + c];
      out[i * d + c] = (float)(acc / denom);
    }
  }
  return 0;
}

}  // extern "C"
