/*
 * CPU oracle for paged GQA decode attention -- TEST INFRASTRUCTURE ONLY.
 *
 * Plain, slow, obviously correct scalar C. Only the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg may load it; the product
 * path never does. It shares no code, header or table with the CUDA library.
 *
 * Sources (web pages on paged attention; citations name page and section):
 *  [TFF]  "十年 C++ 后端 GAP 六个月，写了一个近 3 万行的LLM-TFFInfer推理框架",
 *         section 3.6.4 KVCache (PageManager / LayerKVContext::get_location:
 *         logical token -> (page_table[token / PAGE_SIZE], token % PAGE_SIZE)),
 *         section 3.7.2 item 5 (online softmax).
 *  [HET]  the heterogeneous C++ LLM engine article: section 2.3 (paged
 *         attention: walk the page table, read physical blocks), section 2.4
 *         (int8/uint4 KV with per-channel / per-block scales), section 2.6
 *         (asymmetric per-channel formula: scale = (max-min)/255,
 *         zero_point = round(-min/scale), Q = clamp(round(x/scale)+zp, 0, 255),
 *         dequant (Q - zp) * scale), section 4.3 (paged_attention_kernel:
 *         indirect addressing, dequant, score / sqrt(head_dim), softmax, P.V,
 *         normalise), section 4.4 (two 4-bit values packed per byte).
 *  [QW]   "从零实现 C++ LLM 推理引擎" section "3. GQA": 28 Q heads share 4 KV
 *         heads (repeat_kv), i.e. query head h reads KV head h / (Hq/Hkv).
 *  [OFP8] the E4M3 encoding of the OCP 8-bit floating point specification
 *         (the pages fix no FP8 scheme: TFFInfer section 9.3 lists FP8
 *         among the quantisation formats to add, and the engine article,
 *         section 4.5, notes FP8 support on Ada/Hopper parts).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *  - round() is round-half-to-even (rintf under the default rounding mode).
 *  - zero_point is not clamped and is stored as int32; float->int32
 *    conversions saturate; the code sum is formed in 64-bit then clamped.
 *  - degenerate range: when (max-min)/L is not > 0 the scale is |min|/L, or
 *    1.0 when that is not > 0 either (so one-token blocks round-trip exactly).
 *  - granularity: one (scale, zp) per (physical block, kv head, channel),
 *    separately for K and V; an append into a partly filled block
 *    re-quantises the whole block from the dequantised old values plus the
 *    new bf16 values.
 *  - uint4 packs channel 2j in the low nibble and 2j+1 in the high nibble.
 *  - decode attends to every token t < seq_len (the new token is stored
 *    first); an empty sequence gives a zero output row.
 *  - fp8 KV: E4M3 codes with one symmetric fp32 scale per (physical block,
 *    kv head, channel), separately for K and V (the integer formats'
 *    granularity): scale = max|x| / 448 (1.0 for an all-zero channel),
 *    code = E4M3(x / scale) rounded to nearest-even and saturated to +-448,
 *    the sign kept for zero results; appends re-quantise the whole block as
 *    for the integer formats, from float(value(code)) * scale.
 *  - several query tokens per sequence (chunked prefill, speculative
 *    verification): all of them are stored before the call and query token
 *    i of n_q attends causally to t < seq_len - (n_q - 1 - i).
 *
 * Build: gcc -O2 -ffp-contract=off -fno-fast-math (fp32 steps stay IEEE
 * single operations; the decode is fp64).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define KV_BF16 0
#define KV_UINT8 1
#define KV_UINT4 2
#define KV_FP8 3

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads the OpenMP loops below use from now on (n >= 1); a timing knob for
   the benchmark's CPU baseline, with no effect on any result. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

static float bf16_to_float(uint16_t b) {
  uint32_t u = ((uint32_t)b) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* float -> int32 with saturation; NaN -> 0. x is already integral. */
static int32_t sat_i32(float x) {
  if (x != x) return 0;
  if (x >= 2147483648.0f) return INT32_MAX;
  if (x <= -2147483648.0f) return INT32_MIN;
  return (int32_t)x;
}

/*
 * Quantise one channel of one block ([HET] section 2.6), in IEEE fp32:
 *   mn, mx  = min / max of vals
 *   scale   = (mx - mn) / L                (L = 255 for uint8, 15 for uint4)
 *             degenerate: |mn| / L, or 1.0
 *   zp      = rint(-mn / scale)            (int32, not clamped)
 *   code[i] = clamp(rint(vals[i] / scale) + zp, 0, L)
 */
void oracle_quant_channel(const float* vals, int n, int L, float* scale_out, int32_t* zp_out,
                          int32_t* codes) {
  float mn = vals[0], mx = vals[0];
  for (int i = 1; i < n; ++i) {
    if (vals[i] < mn) mn = vals[i];
    if (vals[i] > mx) mx = vals[i];
  }
  volatile float r = mx - mn;
  volatile float scale = r / (float)L;
  if (!(scale > 0.0f)) {
    volatile float a = fabsf(mn);
    scale = a / (float)L;
    if (!(scale > 0.0f)) scale = 1.0f;
  }
  volatile float zq = -mn / scale;
  int32_t zp = sat_i32(rintf(zq));
  for (int i = 0; i < n; ++i) {
    volatile float xq = vals[i] / scale;
    int64_t c = (int64_t)sat_i32(rintf(xq)) + (int64_t)zp;
    if (c < 0) c = 0;
    if (c > L) c = L;
    codes[i] = (int32_t)c;
  }
  *scale_out = scale;
  *zp_out = zp;
}

/*
 * E4M3 ([OFP8]): 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits,
 * no infinities. Exponent field 15 with mantissa 7 is NaN, so the largest
 * finite magnitude is 1.75 * 2^8 = 448. Exponent field 0 holds the
 * subnormals m/8 * 2^-6 = m * 2^-9.
 */
double oracle_e4m3_value(int code) {
  const int e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
  return (code & 0x80) ? -v : v;
}

/*
 * Finite fp32 -> E4M3: round to nearest, ties to even, magnitudes that
 * round above 448 saturate to 448; the sign is kept (so -0.0 and small
 * negative values give 0x80). Every step is exact in double: a / q only
 * shifts the exponent.
 */
int oracle_e4m3_encode(float y) {
  const int sign = signbit(y) ? 0x80 : 0;
  const double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7E;
  int e;  /* binade [2^e, 2^(e+1)) of a; below 2^-6 the subnormal spacing */
  if (a < ldexp(1.0, -6)) {
    e = -6;
  } else {
    frexp(a, &e);
    e -= 1;
  }
  const double q = ldexp(1.0, e - 3);  /* spacing of the 3-bit mantissa */
  double m = nearbyint(a / q);
  const double v = m * q;              /* may carry into the next binade */
  if (v == 0.0) return sign;
  if (v < ldexp(1.0, -6)) return sign | (int)(v / ldexp(1.0, -9));
  int ev;
  frexp(v, &ev);
  ev -= 1;
  const int mant = (int)(ldexp(v, -ev) * 8.0) - 8;
  return sign | ((ev + 7) << 3) | mant;
}

void oracle_e4m3_encode_array(const float* y, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = (uint8_t)oracle_e4m3_encode(y[i]);
}

/*
 * Quantise one channel of one block to E4M3 with a symmetric scale, in IEEE
 * fp32 (reading in the header):
 *   amax    = max_i |vals[i]|
 *   scale   = amax / 448                (1.0 when not > 0)
 *   code[i] = E4M3(vals[i] / scale)
 */
void oracle_quant_channel_fp8(const float* vals, int n, float* scale_out, int32_t* codes) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    const float a = fabsf(vals[i]);
    if (a > amax) amax = a;
  }
  volatile float scale = amax / 448.0f;
  if (!(scale > 0.0f)) scale = 1.0f;
  for (int i = 0; i < n; ++i) {
    volatile float y = vals[i] / scale;
    codes[i] = oracle_e4m3_encode(y);
  }
  *scale_out = scale;
}

/* stored code of (page, slot, channel) -- page = (phys, kv head) */
static int read_code(int kv_dtype, const uint8_t* codes, int64_t page, int bs, int D, int slot,
                     int c) {
  if (kv_dtype == KV_UINT8 || kv_dtype == KV_FP8) return codes[(page * bs + slot) * D + c];
  uint8_t byte = codes[(page * bs + slot) * (D / 2) + c / 2];
  return (c & 1) ? (byte >> 4) : (byte & 15);
}

static void write_code(int kv_dtype, uint8_t* codes, int64_t page, int bs, int D, int slot, int c,
                       int code) {
  if (kv_dtype == KV_UINT8 || kv_dtype == KV_FP8) {
    codes[(page * bs + slot) * D + c] = (uint8_t)code;
    return;
  }
  uint8_t* p = &codes[(page * bs + slot) * (D / 2) + c / 2];
  if (c & 1)
    *p = (uint8_t)((*p & 0x0F) | (code << 4));
  else
    *p = (uint8_t)((*p & 0xF0) | code);
}

/*
 * Append new tokens to the paged pool ([TFF] section 3.6.4 append_token /
 * get_location; [HET] sections 2.4, 2.6, 4.3). One tensor (K or V) per call.
 *
 * new_bits: bf16 [T_new][Hkv][D]; sequence b's new tokens are rows
 * cu_new[b]..cu_new[b+1] and take logical positions ctx_lens[b]...
 * Pool arrays use the library's storage format:
 *   bf16 : pool16[P][Hkv][bs][D]
 *   uint8: codes[P][Hkv][bs][D], scale[P][Hkv][D], zp[P][Hkv][D]
 *   uint4: codes[P][Hkv][bs][D/2] (low nibble = even channel), scale, zp
 *   fp8  : codes[P][Hkv][bs][D] (E4M3 bits), scale[P][Hkv][D]; zp unused
 * Returns 0, or -1 for a block-table entry outside [0, num_blocks) or a
 * position past max_blocks * bs.
 */
int oracle_append(int kv_dtype, int num_blocks, int Hkv, int bs, int D, uint16_t* pool16,
                  uint8_t* codes, float* scale, int32_t* zp, const uint16_t* new_bits,
                  const int32_t* cu_new, const int32_t* ctx_lens, const int32_t* block_table,
                  int batch, int max_blocks) {
  const int L = (kv_dtype == KV_UINT4) ? 15 : 255;
  float* vals = (float*)malloc(sizeof(float) * (size_t)bs);
  int32_t* qc = (int32_t*)malloc(sizeof(int32_t) * (size_t)bs);
  int status = 0;
  for (int b = 0; b < batch; ++b) {
    const int n_new = cu_new[b + 1] - cu_new[b];
    if (n_new <= 0) continue;
    const int ctx = ctx_lens[b];
    const int total = ctx + n_new;
    if (ctx < 0 || total > max_blocks * bs) {
      status = -1;
      continue;
    }
    for (int blk = ctx / bs; blk <= (total - 1) / bs; ++blk) {
      const int phys = block_table[(int64_t)b * max_blocks + blk];
      if (phys < 0 || phys >= num_blocks) {
        status = -1;
        continue;
      }
      const int first = blk * bs;
      const int old_cnt = ctx > first ? (ctx - first < bs ? ctx - first : bs) : 0;
      const int valid = total - first < bs ? total - first : bs;
      for (int h = 0; h < Hkv; ++h) {
        const int64_t page = (int64_t)phys * Hkv + h;
        for (int c = 0; c < D; ++c) {
          if (kv_dtype == KV_BF16) {
            for (int s = old_cnt; s < valid; ++s) {
              const int64_t row = cu_new[b] + (first + s - ctx);
              pool16[(page * bs + s) * D + c] = new_bits[(row * Hkv + h) * D + c];
            }
            continue;
          }
          const float old_scale = scale[page * D + c];
          if (kv_dtype == KV_FP8) {
            for (int s = 0; s < valid; ++s) {
              if (s < old_cnt) {
                /* stored token: float(value(code)) * scale, one fp32 multiply */
                volatile float f = (float)oracle_e4m3_value(read_code(kv_dtype, codes, page, bs, D, s, c));
                volatile float x = f * old_scale;
                vals[s] = x;
              } else {
                const int64_t row = cu_new[b] + (first + s - ctx);
                vals[s] = bf16_to_float(new_bits[(row * Hkv + h) * D + c]);
              }
            }
            float sc;
            oracle_quant_channel_fp8(vals, valid, &sc, qc);
            for (int s = 0; s < valid; ++s) write_code(kv_dtype, codes, page, bs, D, s, c, qc[s]);
            scale[page * D + c] = sc;
            continue;
          }
          const int32_t old_zp = zp[page * D + c];
          for (int s = 0; s < valid; ++s) {
            if (s < old_cnt) {
              /* stored token: float(code - zp) * scale, one fp32 multiply */
              const int32_t diff = read_code(kv_dtype, codes, page, bs, D, s, c) - old_zp;
              volatile float f = (float)diff;
              volatile float x = f * old_scale;
              vals[s] = x;
            } else {
              const int64_t row = cu_new[b] + (first + s - ctx);
              vals[s] = bf16_to_float(new_bits[(row * Hkv + h) * D + c]);
            }
          }
          float sc;
          int32_t z;
          oracle_quant_channel(vals, valid, L, &sc, &z, qc);
          for (int s = 0; s < valid; ++s) write_code(kv_dtype, codes, page, bs, D, s, c, qc[s]);
          scale[page * D + c] = sc;
          zp[page * D + c] = z;
        }
      }
    }
  }
  free(vals);
  free(qc);
  return status;
}

/* K or V element of token slot `slot` in page `page`, as a double. */
static double kv_value(int kv_dtype, const uint16_t* pool16, const uint8_t* codes,
                       const float* scale, const int32_t* zp, int64_t page, int bs, int D,
                       int slot, int c) {
  if (kv_dtype == KV_BF16) return (double)bf16_to_float(pool16[(page * bs + slot) * D + c]);
  const int code = read_code(kv_dtype, codes, page, bs, D, slot, c);
  if (kv_dtype == KV_FP8) return oracle_e4m3_value(code) * (double)scale[page * D + c];
  return ((double)code - (double)zp[page * D + c]) * (double)scale[page * D + c];
}

/*
 * Attention of one query row over the first n tokens of sequence b
 * ([HET] section 4.3; [QW] "3. GQA"; [TFF] section 3.6.4 addressing), with
 * query head h reading KV head j = h / g:
 *   K_t, V_t  = slot t % bs of physical block block_table[b][t / bs], head j
 *   s_t       = softmax_scale * sum_c q[c] * K_t[c]                  (fp64)
 *   p_t       = exp(s_t - max_t s_t) / sum_t exp(s_t - max_t s_t)    (two-pass)
 *   o[c]      = sum_t p_t * V_t[c]
 * Quantised pools are read through kv_value in fp64. n <= 0 gives a zero
 * row. Returns 0, or -1 (row left as NaN) if n > max_blocks * bs or a
 * block-table entry it reads lies outside [0, num_blocks).
 */
static int attend_row(int kv_dtype, int num_blocks, int Hkv, int bs, int D, const uint16_t* k16,
                      const uint16_t* v16, const uint8_t* kc, const uint8_t* vc, const float* ks,
                      const int32_t* kz, const float* vs, const int32_t* vz, const uint16_t* q,
                      int h, int g, const int32_t* table_row, int max_blocks, int n,
                      double softmax_scale, double* o) {
  const int j = h / g;
  for (int c = 0; c < D; ++c) o[c] = 0.0;
  if (n <= 0) return 0;
  if (n > max_blocks * bs) {
    for (int c = 0; c < D; ++c) o[c] = NAN;
    return -1;
  }
  for (int t = 0; t < n; t += bs) {
    const int phys = table_row[t / bs];
    if (phys < 0 || phys >= num_blocks) {
      for (int c = 0; c < D; ++c) o[c] = NAN;
      return -1;
    }
  }
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  double mx = -INFINITY;
  for (int t = 0; t < n; ++t) {
    const int64_t page = (int64_t)table_row[t / bs] * Hkv + j;
    double acc = 0.0;
    for (int c = 0; c < D; ++c)
      acc += (double)bf16_to_float(q[c]) *
             kv_value(kv_dtype, k16, kc, ks, kz, page, bs, D, t % bs, c);
    s[t] = softmax_scale * acc;
    if (s[t] > mx) mx = s[t];
  }
  double denom = 0.0;
  for (int t = 0; t < n; ++t) {
    s[t] = exp(s[t] - mx);
    denom += s[t];
  }
  for (int t = 0; t < n; ++t) {
    const int64_t page = (int64_t)table_row[t / bs] * Hkv + j;
    const double p = s[t] / denom;
    for (int c = 0; c < D; ++c)
      o[c] += p * kv_value(kv_dtype, v16, vc, vs, vz, page, bs, D, t % bs, c);
  }
  free(s);
  return 0;
}

/*
 * Decode attention for selected rows (b, h): row r = rows[i] has
 * b = r / Hq, h = r % Hq and attends to all n = seq_lens[b] stored tokens
 * (the step's new token is stored first). out is [n_rows][D].
 * Returns 0, or -1 if any row failed its checks (see attend_row).
 */
int oracle_decode(int kv_dtype, int num_blocks, int Hkv, int bs, int D, const uint16_t* k16,
                  const uint16_t* v16, const uint8_t* kc, const uint8_t* vc, const float* ks,
                  const int32_t* kz, const float* vs, const int32_t* vz, const uint16_t* q_bits,
                  int Hq, const int32_t* block_table, const int32_t* seq_lens, int max_blocks,
                  double softmax_scale, const int64_t* rows, int64_t n_rows, double* out) {
  const int g = Hq / Hkv;
  int status = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(min : status)
  for (int64_t i = 0; i < n_rows; ++i) {
    const int64_t r = rows[i];
    const int b = (int)(r / Hq), h = (int)(r % Hq);
    const int st = attend_row(kv_dtype, num_blocks, Hkv, bs, D, k16, v16, kc, vc, ks, kz, vs, vz,
                              q_bits + r * D, h, g, block_table + (int64_t)b * max_blocks,
                              max_blocks, seq_lens[b], softmax_scale, out + i * D);
    if (st < status) status = st;
  }
  return status;
}

/*
 * Attention of several query tokens per sequence over the paged cache
 * (chunked prefill and speculative verification: the engine article,
 * sections 2.2 and 4.2, mixes prefill chunks with decode steps; TFFInfer
 * section 9.3 plans speculative decoding). All n_q new tokens of sequence b
 * are stored before the call, so seq_lens[b] counts them; query token i
 * (0 <= i < n_q) sits at position seq_lens[b] - n_q + i and attends
 * causally to every t <= that position:
 *   n_i = seq_lens[b] - (n_q - 1 - i)      (a zero row when n_i <= 0)
 * q_bits is [B][n_q][Hq][D]; row r = rows[k] is ((b * n_q) + i) * Hq + h.
 * Returns 0, or -1 if any row failed its checks (see attend_row).
 */
int oracle_decode_multi(int kv_dtype, int num_blocks, int Hkv, int bs, int D, const uint16_t* k16,
                        const uint16_t* v16, const uint8_t* kc, const uint8_t* vc, const float* ks,
                        const int32_t* kz, const float* vs, const int32_t* vz,
                        const uint16_t* q_bits, int n_q, int Hq, const int32_t* block_table,
                        const int32_t* seq_lens, int max_blocks, double softmax_scale,
                        const int64_t* rows, int64_t n_rows, double* out) {
  const int g = Hq / Hkv;
  int status = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(min : status)
  for (int64_t k = 0; k < n_rows; ++k) {
    const int64_t r = rows[k];
    const int64_t bi = r / Hq;
    const int h = (int)(r % Hq), b = (int)(bi / n_q), i = (int)(bi % n_q);
    const int n_i = seq_lens[b] - (n_q - 1 - i);
    const int st = attend_row(kv_dtype, num_blocks, Hkv, bs, D, k16, v16, kc, vc, ks, kz, vs, vz,
                              q_bits + r * D, h, g, block_table + (int64_t)b * max_blocks,
                              max_blocks, n_i, softmax_scale, out + k * D);
    if (st < status) status = st;
  }
  return status;
}
