/*
 * kvq.h — C ABI of the quantized KV cache and its fused-dequant decode attention
 * (libkvq.so, CUDA, sm_103a).
 *
 * What it computes
 *   Asymmetric affine quantization of the attention KV cache, as in the page
 *   "KV Cache Quantization — 8-bit and 4-bit", § Integer quantization in one screen:
 *       scale      = (x_max - x_min) / (q_max - q_min)
 *       zero_point = q_min - round(x_min / scale)
 *       q          = round(x / scale) + zero_point          (clamped to [q_min, q_max])
 *       x_hat      = scale * (q - zero_point)
 *   with int8 [-128, 127], int4 [-8, 7] and int2 [-2, 1] codes. Keys are quantized
 *   per channel over groups of k_group consecutive tokens, values per token over
 *   groups of v_group consecutive channels (page "Sub-8-Bit KV Cache Quantization Is
 *   Not a Free Lever for an RDNA4 Agent Swarm", § The cache is two distributions, not
 *   one; and "KV Cache Quantization — 8-bit and 4-bit", § Granularity and § Why keys
 *   and values want different treatment). The newest keys that do not yet fill the
 *   residual window stay binary16 ("Sub-8-Bit …", § What the low-bit numbers actually
 *   cost: a small full-precision residual for the most recent tokens). Decode
 *   attention reads the packed integers and dequantizes them on the fly ("KV Cache
 *   Quantization — 8-bit and 4-bit", § Decode is memory-bound, so smaller is also
 *   faster), with softmax(scale * q . k_hat) . v_hat over every cached token.
 *
 * Arithmetic (bit-exact contract of the quantizer)
 *   All of it in IEEE binary32, round to nearest even, no contraction:
 *   range = x_max - x_min; s32 = max(range / (q_max - q_min), max|x| / (2048 - 2^b));
 *   the stored scale is binary16(s32) rounded toward +infinity; zp = q_min -
 *   rint(x_min / scale), an integer of magnitude <= 2048 and so exact in binary16;
 *   q = clamp(rint(x / scale) + zp). The second term of s32 only matters for a narrow
 *   group far from zero, whose zero point would otherwise exceed the integers binary16
 *   holds exactly; with it |x - x_hat| <= scale/2 holds for every group. A group whose
 *   values are all equal is widened to include 0; an all-zero group gets scale 1.
 *   Codes are stored as u = q - q_min (unsigned, b bits). Keys use b = bits, values
 *   b = v_bits (the same unless v_bits says otherwise: 8-bit keys with
 *   4-bit values is the mixed recipe of "KV Cache Quantization — 8-bit and 4-bit",
 *   § Why keys and values want different treatment).
 *
 * Symmetric per-token int8 scheme (symmetric = 1)
 *   The symmetric quantizer of "KV Cache Quantization — 8-bit and 4-bit", § Symmetric
 *   vs asymmetric (zero point 0, integer range centred on real zero, x_hat = scale * q)
 *   with one scale per token for keys and for values — the per-token int8 cache of
 *   "Sub-8-Bit KV Cache Quantization Is Not a Free Lever for an RDNA4 Agent Swarm",
 *   § The RDNA4 kernel angle: s32 = max|x| / 127 over the token's d channels; the stored
 *   scale is binary16(s32) rounded toward +infinity (an all-zero token gets scale 1);
 *   q = clamp(rint(x / scale), -128, 127), stored as u = q + 128. There is no residual
 *   window: every token's keys are quantized when it is appended.
 *   Outlier isolation (k_outliers = k > 0; dense-and-sparse quantization, "Sub-8-Bit …",
 *   § What the low-bit numbers actually cost and § The RDNA4 kernel angle): before a key
 *   row is quantized, its k entries farthest from the row's lower median (the 64th
 *   smallest of the d = 128 values) in binary32 |x - median|, in order of decreasing
 *   distance with ties to the lower channel, are stored as (channel, binary16 value)
 *   and replaced by 0; k_hat is the dense x_hat plus those values at their channels.
 *   The asymmetric scheme takes the same per-row split (gqa_ratio <= 4): a key row is
 *   split when its token leaves the binary16 residual window, and the per-channel
 *   groups are then formed over the dense rows (the isolated entries read as 0 there).
 *   Residual rows are exact binary16 copies and carry no entries.
 *
 * State after T tokens of one (layer, batch row, kv head)
 *   R_eff = residual_len, or k_group when residual_len == 0.
 *   Keys of tokens [0, Tq), Tq = floor(T / R_eff) * R_eff, are quantized; keys of
 *   tokens [Tq, T) are binary16 copies in residual slot (t mod R_eff). Values of all
 *   T tokens are quantized. The state depends only on the token history, never on
 *   how the tokens were split into append calls.
 *
 * Memory (all device memory, owned by the caller; this library allocates nothing)
 *   S_pad = max_seq_len rounded up to a multiple of 128; LBH = n_layers*batch*n_kv_heads;
 *   slices are ordered [layer][batch][kv head]. Per slice:
 *     k_codes : S_pad rows of d*b/8 bytes. Channel c occupies bits [c*b, c*b+b) of its
 *               row (little-endian bytes, low bits first).
 *     k_meta  : (S_pad / k_group) groups x d channels x {scale, zero_point} binary16,
 *               followed when k_outliers = k > 0 by S_pad x k entries {channel (uint16),
 *               value (binary16)} (entries of tokens >= Tq are undefined).
 *     k_resid : R_eff rows of d binary16.
 *     v_codes : S_pad/2 pair rows of 2*d*b_v/8 bytes (b_v = value code width). Channel c of a token sits at
 *               position pos(c) = (d/8)*(c%8) + 2*(c/16) + (c/8)%2 of that token's
 *               d*b_v/8-byte row; the rows of tokens 2p and 2p+1 are interleaved in
 *               16-bit units (32-bit word k of pair row p = unit k of token 2p in the
 *               low half, unit k of token 2p+1 in the high half).
 *     v_meta  : S_pad/2 token pairs x (d / v_group) groups x a record of four binary16
 *               values {scale of token 2p, scale of token 2p+1, zero point of token 2p,
 *               zero point of token 2p+1} (8 bytes; 4 bytes per token and group).
 *   Symmetric scheme: k_codes and v_codes as above (b = 8); k_meta is S_pad binary16 key
 *   scales (one per token), followed when k_outliers = k > 0 by S_pad x k entries
 *   {channel (uint16), value (binary16)}; v_meta holds the pair records of one value
 *   group per token (v_group == d) with zero points +0; there is no k_resid (its size is
 *   0 and its pointer may be NULL).
 *   Every buffer must be 256-byte aligned (torch and cudaMalloc allocations are) and
 *   zero-filled before the first append.
 *
 * Calls
 *   Every call checks its arguments on the host first and launches nothing when they
 *   are wrong. Work is enqueued asynchronously on `stream` (a cudaStream_t; NULL is
 *   the legacy default stream); nothing synchronizes. Functions keep no state and are
 *   reentrant; calls that touch the same buffers must be ordered by the caller.
 *   A launch failure is reported as KVQ_ERR_CUDA (cudaGetLastError after the launch).
 */
#ifndef KVQ_H_
#define KVQ_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KVQ_OK = 0,
  KVQ_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad layer, s_cur/n_new out of order */
  KVQ_ERR_UNSUPPORTED = 2, /* a configuration this build does not implement */
  KVQ_ERR_CAPACITY = 3,    /* s_cur + n_new > max_seq_len */
  KVQ_ERR_WORKSPACE = 4,   /* decode workspace missing or too small */
  KVQ_ERR_CUDA = 5         /* a CUDA launch reported an error */
} kvq_status;

/* Cache shape and quantizer settings; the names follow the pages' problem
 * statement ("KV Cache Quantization — 8-bit and 4-bit", § The bytes-per-token
 * formula: L, n_kv, d_head, S). Supported: d_head == 128; bits in {2, 4, 8};
 * v_bits == 0 (same as bits) or v_bits == bits, or bits == 8 with v_bits == 4;
 * k_group and v_group in {32, 64, 128}; residual_len == 0 or a multiple of k_group
 * up to 1024; 1 <= gqa_ratio <= 8; n_kv_heads <= 255; batch <= 4095;
 * 1 <= max_seq_len <= 2^24. symmetric == 1 needs bits == 8, v_bits in {0, 8},
 * v_group == d_head and residual_len == 0 (k_group is then unused but must still be
 * one of the values above); k_outliers in 0..4, and > 0 with symmetric == 0 only when
 * gqa_ratio <= 4. */
typedef struct {
  int32_t n_layers;     /* L */
  int32_t batch;        /* B: sequences; all share one length */
  int32_t n_kv_heads;   /* n_kv */
  int32_t gqa_ratio;    /* r: query heads per kv head; query head i reads kv head i / r */
  int32_t d_head;       /* d */
  int32_t max_seq_len;  /* capacity in tokens */
  int32_t bits;         /* b: code width of the keys (and of the values when v_bits == 0) */
  int32_t k_group;      /* G: tokens per key group (keys are quantized per channel) */
  int32_t v_group;      /* Gv: channels per value group (values are quantized per token) */
  int32_t residual_len; /* R: binary16 key residual capacity; 0 means k_group */
  int32_t v_bits;       /* value code width; 0 means bits */
  int32_t symmetric;    /* 0: asymmetric (above); 1: symmetric per-token int8 keys and values */
  int32_t k_outliers;   /* key entries per token kept in a sparse side list (0..4) */
} kvq_config;

/* Device pointers to the five cache buffers of all layers (layout above). */
typedef struct {
  void* k_codes;
  void* k_meta;
  void* k_resid;
  void* v_codes;
  void* v_meta;
} kvq_buffers;

enum { KVQ_BUF_K_CODES = 0, KVQ_BUF_K_META = 1, KVQ_BUF_K_RESID = 2, KVQ_BUF_V_CODES = 3, KVQ_BUF_V_META = 4,
       KVQ_NUM_BUFFERS = 5 };

/* Sizes in bytes of the five buffers for `cfg` (layout above), so that the caller can
 * allocate them. Returns KVQ_ERR_INVALID_ARG / KVQ_ERR_UNSUPPORTED for a bad config. */
kvq_status kvq_buffer_sizes(const kvq_config* cfg, size_t bytes[KVQ_NUM_BUFFERS]);

/* Append n_new >= 1 tokens of one layer after the s_cur tokens already cached
 * (s_cur + n_new <= max_seq_len). k_f16 and v_f16 are device binary16 arrays
 * [batch][n_new][n_kv_heads][d_head] (16-byte aligned). Values are quantized per token;
 * keys go to the residual window and every residual window that fills is quantized
 * per channel (its R_eff / k_group groups at once). A prefill is s_cur = 0,
 * n_new = prompt length; a decode step is n_new = 1. */
kvq_status kvq_quantize_append(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                               int64_t n_new, const void* k_f16, const void* v_f16, void* stream);

/* Dequantize the first s_cur tokens of one layer into binary32 arrays
 * k_out, v_out [batch][n_kv_heads][s_cur][d_head] (device, 16-byte aligned):
 * x_hat = scale * (q - zero_point) as one binary32 product; residual keys are copied.
 * For tests and inspection: the decode path never materializes these. */
kvq_status kvq_dequantize(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                          float* k_out, float* v_out, void* stream);

/* Bytes of device workspace kvq_decode_attention needs for s_cur cached tokens
 * (0 for a bad config). The workspace holds an error word (first 4 bytes, see
 * kvq_decode_error), per-(batch, kv head) counters and split-K partials; zero-fill it
 * once before its first use: every call leaves the counters at zero again. */
size_t kvq_decode_workspace_size(const kvq_config* cfg, int64_t s_cur);

/* Decode attention of one layer over its s_cur >= 1 cached tokens (the token just
 * appended included). q_f16 [batch][n_kv_heads*gqa_ratio][d_head] binary16, out the
 * same shape in binary32 (device, 16-byte aligned):
 *   out[b][i] = sum_t softmax_t(softmax_scale * q[b][i] . k_hat[t]) * v_hat[t]
 * with k_hat / v_hat of kv head i / gqa_ratio, dequantized on the fly. ws/ws_bytes:
 * workspace of at least kvq_decode_workspace_size(cfg, s_cur) bytes. */
kvq_status kvq_decode_attention(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                                const void* q_f16, float softmax_scale, float* out, void* ws, size_t ws_bytes,
                                void* stream);

/* One decode step of one layer: exactly kvq_quantize_append(cfg, bufs, layer, s_cur, 1,
 * k_f16, v_f16, stream) followed by kvq_decode_attention over s_cur + 1 tokens, in one
 * kernel launch when the new token does not fill a residual window (the CTA whose
 * token range holds the new token appends it before reading its stages), and in the
 * two launches otherwise. k_f16, v_f16: [batch][1][n_kv_heads][d_head] binary16
 * (16-byte aligned). Same cache state and outputs as the two calls ("KV Cache
 * Quantization — 8-bit and 4-bit", § Decode is memory-bound, so smaller is also
 * faster: one pass over the cache per step). In the symmetric scheme (no residual
 * window) it is always one launch. */
kvq_status kvq_decode_step(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                           const void* k_f16, const void* v_f16, const void* q_f16, float softmax_scale, float* out,
                           void* ws, size_t ws_bytes, void* stream);

/* Flag bits of kvq_decode_attention_ex and kvq_decode_step_ex (other bits:
 * KVQ_ERR_INVALID_ARG).
 * KVQ_DECODE_EARLY_PREFETCH: the tensor-core kernel starts copying this layer's cache
 * tiles before the kernel launched just before it on `stream` has finished (with
 * programmatic dependent launch the two overlap: this launch's first tiles stream in
 * while the previous one merges its partials). The caller guarantees that this previous
 * kernel writes no cache memory of `layer`; kernels before it have finished by then,
 * because every launch of this library waits for its predecessor before it lets the
 * next one start. Decode steps that visit the layers of a model in turn (n_layers > 1)
 * meet the condition; a step that directly follows kvq_quantize_append or
 * kvq_decode_step of the same layer does not. Queries and new key/value rows are always
 * read after the wait. No counterpart in the pages: a scheduling choice of this library. */
#define KVQ_DECODE_EARLY_PREFETCH 1u
/* KVQ_DECODE_ZERO_WAIT_LIMIT: the tensor-core kernel's bounded waits for its staged cache
 * tiles get a time limit of 0 (normally about 2 s of the GPU's global timer): every
 * CTA gives up at its first wait, drains the copies it has in flight, records
 * KVQ_DECODE_ERR_WAIT_TIMEOUT in the workspace error word and finishes, so the
 * outputs of that call are undefined. For testing the failure path: nothing faults or
 * hangs, and the context stays usable. */
#define KVQ_DECODE_ZERO_WAIT_LIMIT 2u

/* Bits of the decode error word (kvq_decode_error). */
#define KVQ_DECODE_ERR_WAIT_TIMEOUT 1u /* a wait for staged cache tiles ran out of time */

/* kvq_decode_attention with flag bits (0: identical to kvq_decode_attention). */
kvq_status kvq_decode_attention_ex(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                                   const void* q_f16, float softmax_scale, float* out, void* ws, size_t ws_bytes,
                                   void* stream, uint32_t flags);

/* kvq_decode_step with flag bits (0: identical to kvq_decode_step). When the step takes
 * two launches (the new token fills a residual window) the flag applies to neither: the
 * attention launch reads what the append launch before it wrote. */
kvq_status kvq_decode_step_ex(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                              const void* k_f16, const void* v_f16, const void* q_f16, float softmax_scale,
                              float* out, void* ws, size_t ws_bytes, void* stream, uint32_t flags);

/* Device-side status of decode launches. The tensor-core kernel bounds every wait for
 * its staged cache tiles; a wait that runs out sets KVQ_DECODE_ERR_WAIT_TIMEOUT in the
 * error word (the first 4 bytes of the workspace `ws`), and the outputs of that launch
 * are then not to be trusted, although the call returned KVQ_OK. This call waits until
 * every launch enqueued before it on `stream` has finished (it synchronizes the
 * stream), stores the word in *err_out (0: no error since the last read) and clears
 * it. ws_bytes: the workspace size (at least 256). Returns KVQ_ERR_WORKSPACE for a
 * missing or misaligned workspace, KVQ_ERR_CUDA if the copy fails. */
kvq_status kvq_decode_error(void* ws, size_t ws_bytes, void* stream, uint32_t* err_out);

/* Kernel choice for kvq_decode_attention_impl. AUTO is what kvq_decode_attention uses. */
typedef enum {
  KVQ_DECODE_AUTO = 0,
  KVQ_DECODE_SIMT = 1, /* binary32 CUDA-core dot products (asymmetric, equal code widths only) */
  KVQ_DECODE_MMA = 2   /* tensor-core m16n8k16 products over exact integer codes */
} kvq_decode_impl;

/* kvq_decode_attention with an explicit kernel choice (for comparison runs). */
kvq_status kvq_decode_attention_impl(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                                     const void* q_f16, float softmax_scale, float* out, void* ws,
                                     size_t ws_bytes, void* stream, kvq_decode_impl impl);

/* kvq_decode_attention without a caller-supplied workspace, for callers that cannot
 * allocate device memory at the call site (code embedded in a framework whose allocator
 * owns all device memory, or a decode loop where an allocation's implicit device
 * synchronisation is not acceptable). No counterpart in the pages: it is a deployment
 * convenience of this library. The split-K scratch is one file-scope __device__ array
 * of 16 MiB that every GPU loading the library keeps until the process exits; a
 * configuration whose kvq_decode_workspace_size(cfg, s_cur) exceeds 16 MiB is rejected
 * with KVQ_ERR_WORKSPACE. The function allocates nothing (no cudaMalloc/cudaFree, no
 * allocating library call). Its first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current; make that first call before
 * any stream capture. Every call on a device shares the one array: it clears the
 * array's counters and error word on `stream` (after all its argument checks, so a
 * rejected call writes nothing) and then runs the same kernels as kvq_decode_attention,
 * so calls whose executions overlap on the GPU (other streams, other threads) race and
 * must be ordered by the caller. The looked-up address is kept per device for the life
 * of the process; it does not survive cudaDeviceReset. */
kvq_status kvq_decode_attention_noalloc(const kvq_config* cfg, const kvq_buffers* bufs, int32_t layer, int64_t s_cur,
                                        const void* q_f16, float softmax_scale, float* out, void* stream);

/* kvq_decode_error for the static array of kvq_decode_attention_noalloc on the current
 * device: the error word of the last noalloc call (each call clears it first). Like
 * that call it allocates nothing; it synchronizes `stream`. */
kvq_status kvq_decode_noalloc_error(void* stream, uint32_t* err_out);

/* Number of split-K partitions kvq_decode_attention gives a (batch row, kv head) pair
 * for s_cur tokens (>= 1; when pairs get different counts, the largest), or 0 for a bad
 * config. */
int32_t kvq_decode_num_splits(const kvq_config* cfg, int64_t s_cur);

/* Human-readable name of a status code (static string). */
const char* kvq_status_string(kvq_status status);

/* Library version, e.g. "kvq 0.1.0 sm_103a". */
const char* kvq_version(void);

#ifdef __cplusplus
}
#endif

#endif /* KVQ_H_ */
