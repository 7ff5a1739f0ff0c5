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

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
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

/* stored code of (page, slot, channel) -- page = (phys, kv head) */
static int read_code(int kv_dtype, const uint8_t* codes, int64_t page, int bs, int D, int slot,
                     int c) {
  if (kv_dtype == KV_UINT8) return codes[(page * bs + slot) * D + c];
  uint8_t byte = codes[(page * bs + slot) * (D / 2) + c / 2];
  return (c & 1) ? (byte >> 4) : (byte & 15);
}

static void write_code(int kv_dtype, uint8_t* codes, int64_t page, int bs, int D, int slot, int c,
                       int code) {
  if (kv_dtype == KV_UINT8) {
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
  return ((double)code - (double)zp[page * D + c]) * (double)scale[page * D + c];
}

/*
 * Decode attention for selected rows (b, h) ([HET] section 4.3; [QW] "3. GQA";
 * [TFF] section 3.6.4 addressing). For row r = rows[i] with b = r / Hq,
 * h = r % Hq, j = h / (Hq / Hkv) and n = seq_lens[b]:
 *   K_t, V_t  = slot t % bs of physical block block_table[b][t / bs], head j
 *   s_t       = softmax_scale * sum_c q[b][h][c] * K_t[c]            (fp64)
 *   p_t       = exp(s_t - max_t s_t) / sum_t exp(s_t - max_t s_t)    (two-pass)
 *   out[i][c] = sum_t p_t * V_t[c]
 * Quantised pools are read as (code - zp) * scale in fp64. n == 0 gives a
 * zero row. Returns 0, or -1 if any row touches a block-table entry outside
 * [0, num_blocks) or n > max_blocks * bs (that row is left as NaN).
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
    const int b = (int)(r / Hq), h = (int)(r % Hq), j = h / g;
    const int n = seq_lens[b];
    double* o = out + i * D;
    for (int c = 0; c < D; ++c) o[c] = 0.0;
    if (n <= 0) continue;
    if (n > max_blocks * bs) {
      for (int c = 0; c < D; ++c) o[c] = NAN;
      status = -1;
      continue;
    }
    int bad = 0;
    for (int t = 0; t < n; t += bs) {
      const int phys = block_table[(int64_t)b * max_blocks + t / bs];
      if (phys < 0 || phys >= num_blocks) bad = 1;
    }
    if (bad) {
      for (int c = 0; c < D; ++c) o[c] = NAN;
      status = -1;
      continue;
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    const uint16_t* q = q_bits + ((int64_t)b * Hq + h) * D;
    double mx = -INFINITY;
    for (int t = 0; t < n; ++t) {
      const int64_t page = (int64_t)block_table[(int64_t)b * max_blocks + t / bs] * Hkv + j;
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
      const int64_t page = (int64_t)block_table[(int64_t)b * max_blocks + t / bs] * Hkv + j;
      const double p = s[t] / denom;
      for (int c = 0; c < D; ++c)
        o[c] += p * kv_value(kv_dtype, v16, vc, vs, vz, page, bs, D, t % bs, c);
    }
    free(s);
  }
  return status;
}
