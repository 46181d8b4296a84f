/*
 * kvp_oracle.c -- CPU oracle for the paged-KV-cache decode path.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain, obviously correct
 * reference that the CUDA library is checked against.  It shares no code,
 * header, table or helper with the library under pagedattention_decode_kvp_gb300/,
 * and it must never be reached from the product path: only tests/,
 * __graft_entry__.smoke() and the CPU-baseline leg of bench.py load it.
 *
 * Pages cited (titles as they appear, with section):
 *   [ATB-KV]  "ATB KV Cache management" article -- sections "KV Cache 的显存需求"
 *             (memory of the KV cache), "Paged KV Cache" (16-token blocks),
 *             "BlockManager 的调度".
 *   [OPT]     "KV Cache 优化与显存管理" -- section 二 (PagedAttention, MQA/GQA,
 *             INT8/FP8 quantisation) and section 三 (KVCacheQuantizer listing).
 *   [ATB-PA]  "ATB PagedAttention" article -- sections "ATB 的 PagedAttention 实现"
 *             (page table, logical->physical offset), "PagedAttention 的 Attention
 *             计算修改" (standard attention loop, per-page kernel), "踩坑三"
 *             (copy-on-write of a shared page).
 *
 * Everything floating point is computed in IEEE double, except the INT8
 * quantiser, whose arithmetic the [OPT] listing fixes in float32.
 */
#include <fenv.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* element kinds of a cache pool or of q */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_I8 = 2, ORC_E4M3 = 3 };

/* ---------------------------------------------------------------------------
 * Exact widening of the two 16-bit float formats to double.
 * binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits (IEEE 754-2008).
 * bfloat16: the upper 16 bits of an IEEE binary32.
 * ------------------------------------------------------------------------- */
double orc_f16_to_f64(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else if (e == 31) {
    v = (m == 0) ? INFINITY : NAN;
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1.m) * 2^(e-15) */
  }
  return sign ? -v : v;
}

double orc_bf16_to_f64(uint16_t h) {
  uint32_t bits = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent (bias 7), 3 fraction bits;
 * exponent 0 is subnormal (m * 2^-9); S.1111.111 is NaN; there is no infinity;
 * the largest finite magnitude is 1.75 * 2^8 = 448. */
double orc_e4m3_to_f64(uint8_t c) {
  int sign = (c >> 7) & 1;
  int e = (c >> 3) & 0xf;
  int m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) v = ldexp((double)m, -9);
  else v = ldexp((double)(8 + m), e - 10);
  return sign ? -v : v;
}

/* Round a float to the nearest E4M3 value, ties to the even code (even
 * fraction), magnitudes beyond 448 saturating to 448 ("satfinite"); NaN stays
 * NaN.  The 127 non-negative finite codes are increasing in value, so the two
 * neighbours of |x| are found by bisection over the codes. */
uint8_t orc_f32_to_e4m3(float x) {
  if (isnan(x)) return 0x7f;
  uint8_t sign = signbit(x) ? 0x80 : 0x00;
  double a = fabs((double)x);
  if (a >= 448.0) return sign | 0x7e;
  int lo = 0, hi = 0x7e; /* value(lo) <= a < value(hi) */
  while (hi - lo > 1) {
    int mid = (lo + hi) / 2;
    if (orc_e4m3_to_f64((uint8_t)mid) <= a) lo = mid; else hi = mid;
  }
  double vl = orc_e4m3_to_f64((uint8_t)lo), vh = orc_e4m3_to_f64((uint8_t)hi);
  int code;
  if (a - vl < vh - a) code = lo;
  else if (a - vl > vh - a) code = hi;
  else code = (lo % 2 == 0) ? lo : hi;
  return sign | (uint8_t)code;
}

static double load_elem(const void* base, size_t idx, int kind) {
  switch (kind) {
    case ORC_F16: return orc_f16_to_f64(((const uint16_t*)base)[idx]);
    case ORC_BF16: return orc_bf16_to_f64(((const uint16_t*)base)[idx]);
    case ORC_E4M3: return orc_e4m3_to_f64(((const uint8_t*)base)[idx]);
    default: return (double)((const int8_t*)base)[idx];
  }
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ---------------------------------------------------------------------------
 * Decode attention through the block table.
 *
 * [ATB-PA] "PagedAttention 的 Attention 计算修改": the standard loop scores the
 * query against every cached key, exponentiates and weights V; the paged form
 * only changes where key/value i lives.  [ATB-PA] "ATB 的 PagedAttention 实现":
 * logical position i lives in page table entry i / page_size at offset
 * i % page_size.  [ATB-KV] "Paged KV Cache": a page (block) holds 16 tokens.
 * [OPT] 二: grouped-query attention shares one K/V head among a group of query
 * heads; query head h reads K/V head h / (Hq / Hkv) (contiguous groups).
 *
 * For each requested row (b, h), with n = context_lens[b] and g = h / (Hq/Hkv):
 *   K_i = Kc[block_tables[b][i / bs], g, i % bs, :]   (and V_i likewise)
 *   s_i = scale * sum_d q[b,h,d] * K_i[d]
 *   p   = softmax(s)           (subtract max, exp, divide by the sum)
 *   out = sum_i p_i * V_i
 * INT8 and FP8 pools hold codes; the value is code * scale_pool[blk, g, off]
 * ([OPT] 三, dequantize multiplies the code by its scale; FP8 codes are first
 * widened exactly).  n == 0 gives a zero row.
 *
 * rows: [n_rows, 2] (b, h) pairs, or NULL for every (b, h) in order.
 * out:  [n_rows, D] doubles.
 * Returns 0, or -1 if a referenced block id lies outside [0, num_blocks) or
 * n exceeds max_blocks * bs, or -2 on allocation failure.
 * ------------------------------------------------------------------------- */
int orc_attention_decode(double* out, const int32_t* rows, int n_rows,
                         const void* q, int q_kind,
                         const void* k_cache, const void* v_cache, int cache_kind,
                         const float* k_scale, const float* v_scale,
                         const int32_t* block_tables, int max_blocks,
                         const int32_t* context_lens,
                         int B, int Hq, int Hkv, int D, int num_blocks, int bs,
                         double scale) {
  int total = rows ? n_rows : B * Hq;
  int group = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(min : err)
  for (int r = 0; r < total; ++r) {
    int b = rows ? rows[2 * r] : r / Hq;
    int h = rows ? rows[2 * r + 1] : r % Hq;
    int g = h / group;
    int n = context_lens[b];
    double* o = out + (size_t)r * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (n <= 0) continue;
    if (n > max_blocks * bs) { err = -1; continue; }

    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    if (!qv || !s) { free(qv); free(s); err = -2; continue; }
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, ((size_t)b * Hq + h) * D + d, q_kind);

    int bad = 0;
    /* scores */
    for (int i = 0; i < n && !bad; ++i) {
      int blk = block_tables[(size_t)b * max_blocks + i / bs];
      int off = i % bs;
      if (blk < 0 || blk >= num_blocks) { bad = 1; break; }
      size_t row = (((size_t)blk * Hkv + g) * bs + off);
      double kscale = (cache_kind >= ORC_I8) ? (double)k_scale[row] : 1.0;
      double acc = 0.0;
      for (int d = 0; d < D; ++d)
        acc += qv[d] * (load_elem(k_cache, row * D + d, cache_kind) * kscale);
      s[i] = scale * acc;
    }
    if (bad) { err = -1; free(qv); free(s); continue; }
    /* softmax */
    double m = s[0];
    for (int i = 1; i < n; ++i) if (s[i] > m) m = s[i];
    double sum = 0.0;
    for (int i = 0; i < n; ++i) { s[i] = exp(s[i] - m); sum += s[i]; }
    for (int i = 0; i < n; ++i) s[i] /= sum;
    /* weighted values */
    for (int i = 0; i < n; ++i) {
      int blk = block_tables[(size_t)b * max_blocks + i / bs];
      int off = i % bs;
      size_t row = (((size_t)blk * Hkv + g) * bs + off);
      double vscale = (cache_kind >= ORC_I8) ? (double)v_scale[row] : 1.0;
      for (int d = 0; d < D; ++d)
        o[d] += s[i] * (load_elem(v_cache, row * D + d, cache_kind) * vscale);
    }
    free(qv);
    free(s);
  }
  return err;
}

/* ---------------------------------------------------------------------------
 * Append: scatter each new token's K (or V) rows into its slot.
 * [OPT] 三 write_page writes a token's data at (page, offset); [ATB-PA] "踩坑三"
 * WriteKV writes the new token into its page; the slot of a token is
 * block * bs + offset ([ATB-PA] logical->physical: page = pos / size,
 * offset = pos % size).  A negative slot is a padding token and is skipped.
 * src: [T, Hkv, D] elements of elem_bytes; cache: [NB, Hkv, bs, D].
 * Returns 0, or -1 if a slot is >= num_blocks * bs (nothing written for it).
 * ------------------------------------------------------------------------- */
int orc_append(void* cache, const void* src, const int32_t* slot_mapping, int T,
               int Hkv, int D, int elem_bytes, int num_blocks, int bs) {
  int err = 0;
  size_t row_bytes = (size_t)D * elem_bytes;
  for (int t = 0; t < T; ++t) {
    int slot = slot_mapping[t];
    if (slot < 0) continue;
    if ((long long)slot >= (long long)num_blocks * bs) { err = -1; continue; }
    int blk = slot / bs, off = slot % bs;
    for (int h = 0; h < Hkv; ++h) {
      size_t dst_row = ((size_t)blk * Hkv + h) * bs + off;
      size_t src_row = (size_t)t * Hkv + h;
      memcpy((char*)cache + dst_row * row_bytes, (const char*)src + src_row * row_bytes,
             row_bytes);
    }
  }
  return err;
}

/* ---------------------------------------------------------------------------
 * Copy whole blocks: [ATB-PA] "踩坑三" ExtendKVPage copies an entire shared page
 * into a fresh one before writing to it (copy-on-write).
 * pairs: [P, 2] (src, dst) block ids, applied in order.  block_bytes is the size
 * of one block in this pool (Hkv * bs * D * elem_bytes, or Hkv * bs * 4 for a
 * scale pool).  Returns 0, or -1 if an id is outside [0, num_blocks) (pair skipped).
 * ------------------------------------------------------------------------- */
int orc_copy_blocks(void* cache, const int32_t* pairs, int P, size_t block_bytes,
                    int num_blocks) {
  int err = 0;
  for (int p = 0; p < P; ++p) {
    int src = pairs[2 * p], dst = pairs[2 * p + 1];
    if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { err = -1; continue; }
    if (src == dst) continue;
    memcpy((char*)cache + (size_t)dst * block_bytes, (const char*)cache + (size_t)src * block_bytes,
           block_bytes);
  }
  return err;
}

/* ---------------------------------------------------------------------------
 * INT8 quantiser, per token and per head ([OPT] 三, KVCacheQuantizer, the
 * per-channel branch: the abs-max is taken over the last axis, which for rows
 * of shape [D] is one scale per (token, head)).  In float32:
 *   x     = float(src row)                   (exact widening)
 *   amax  = max_j |x_j|
 *   scale = amax / 127                       (IEEE float division)
 *   scale = scale > 0 ? scale : 1            (an all-zero row keeps scale 1)
 *   q_j   = clip(round_half_even(x_j / scale), -128, 127)
 * (NumPy's round is half-to-even, as is nearbyintf under FE_TONEAREST.)
 * src: [rows, D] 16-bit elements of src_kind; q: [rows, D]; scale: [rows].
 * ------------------------------------------------------------------------- */
void orc_quantize_int8(const uint16_t* src, int src_kind, long long rows, int D,
                       int8_t* q, float* scale_out) {
  /* round-half-even is the default IEEE rounding mode; nearbyintf honours it.
   * The floating-point environment is per thread, so each worker sets it. */
#pragma omp parallel
  {
    fesetround(FE_TONEAREST);
#pragma omp for schedule(static)
    for (long long r = 0; r < rows; ++r) {
      const uint16_t* x16 = src + (size_t)r * D;
      float amax = 0.0f;
      for (int j = 0; j < D; ++j) {
        float x = (float)(src_kind == ORC_BF16 ? orc_bf16_to_f64(x16[j]) : orc_f16_to_f64(x16[j]));
        float a = fabsf(x);
        if (a > amax) amax = a;
      }
      volatile float s = amax / 127.0f; /* a float32 division */
      float sc = (s > 0.0f) ? s : 1.0f;
      for (int j = 0; j < D; ++j) {
        float x = (float)(src_kind == ORC_BF16 ? orc_bf16_to_f64(x16[j]) : orc_f16_to_f64(x16[j]));
        volatile float ratio = x / sc;
        float rq = nearbyintf(ratio);
        if (rq > 127.0f) rq = 127.0f;
        if (rq < -128.0f) rq = -128.0f;
        q[(size_t)r * D + j] = (int8_t)rq;
      }
      scale_out[r] = sc;
    }
  }
}

/* ---------------------------------------------------------------------------
 * Per-tensor INT8 quantisation with a given scale ([OPT] 三, the per_tensor
 * branch: one scale for the whole tensor; a paged cache that appends token by
 * token fixes that scale ahead, so it is an input here):
 *   q_j = clip(round_half_even(x_j / scale), -128, 127) in float32.
 * ------------------------------------------------------------------------- */
void orc_quantize_int8_fixed(const uint16_t* src, int src_kind, long long n, float scale,
                             int8_t* q) {
#pragma omp parallel
  {
    fesetround(FE_TONEAREST);
#pragma omp for schedule(static)
    for (long long i = 0; i < n; ++i) {
      float x = (float)(src_kind == ORC_BF16 ? orc_bf16_to_f64(src[i]) : orc_f16_to_f64(src[i]));
      volatile float ratio = x / scale;
      float rq = nearbyintf(ratio);
      if (rq > 127.0f) rq = 127.0f;
      if (rq < -128.0f) rq = -128.0f;
      q[i] = (int8_t)rq;
    }
  }
}

/* ---------------------------------------------------------------------------
 * FP8 (E4M3) quantiser, per token and per head ([OPT] 二: K/V quantised from
 * FP16 to INT8 or FP8).  The pages give the INT8 rule only; the FP8 rule here
 * is the same with the format's largest magnitude in place of 127:
 *   scale = amax / 448 (float32 division; 1 if not > 0),
 *   code  = E4M3 round-to-nearest-even of the float32 quotient x / scale,
 *           saturating at 448.
 * ------------------------------------------------------------------------- */
void orc_quantize_fp8(const uint16_t* src, int src_kind, long long rows, int D, uint8_t* q,
                      float* scale_out) {
  /* the float32 divisions round to nearest-even, as in the INT8 quantisers;
   * the floating-point environment is per thread, so each worker sets it */
#pragma omp parallel
  {
    fesetround(FE_TONEAREST);
#pragma omp for schedule(static)
    for (long long r = 0; r < rows; ++r) {
      const uint16_t* x16 = src + (size_t)r * D;
      float amax = 0.0f;
      for (int j = 0; j < D; ++j) {
        float x = (float)(src_kind == ORC_BF16 ? orc_bf16_to_f64(x16[j]) : orc_f16_to_f64(x16[j]));
        float a = fabsf(x);
        if (a > amax) amax = a;
      }
      volatile float s = amax / 448.0f;
      float sc = (s > 0.0f) ? s : 1.0f;
      for (int j = 0; j < D; ++j) {
        float x = (float)(src_kind == ORC_BF16 ? orc_bf16_to_f64(x16[j]) : orc_f16_to_f64(x16[j]));
        volatile float ratio = x / sc;
        q[(size_t)r * D + j] = orc_f32_to_e4m3(ratio);
      }
      scale_out[r] = sc;
    }
  }
}

/* ---------------------------------------------------------------------------
 * Multi-query paged attention (prefill / chunked prefill).  ([ATB-KV]
 * "Prefix Caching": requests sharing a system prompt reuse its cached K/V;
 * the new part of each request is computed against it.)  Request b holds
 * n = context_lens[b] tokens, the last L = query_start[b+1] - query_start[b]
 * of which are this chunk's queries (their K/V already appended).  Query i of
 * the chunk (global row query_start[b] + i) sits at position n - L + i and
 * attends causally to positions 0 .. n - L + i: the decode definition above
 * with the context cut at that position.
 * rows: [n_rows, 2] (global query row, query head) pairs to compute.
 * Returns 0, -1 on a bad block id / length (L > n, n > max_blocks * bs).
 * ------------------------------------------------------------------------- */
int orc_attention_prefill(double* out, const int32_t* rows, int n_rows, const void* q, int q_kind,
                          const void* k_cache, const void* v_cache, int cache_kind,
                          const int32_t* block_tables, int max_blocks,
                          const int32_t* context_lens, const int32_t* query_start, int B,
                          int Hq, int Hkv, int D, int num_blocks, int bs, double scale) {
  int group = Hq / Hkv;
  int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(min : err)
  for (int r = 0; r < n_rows; ++r) {
    int t = rows[2 * r], h = rows[2 * r + 1];
    double* o = out + (size_t)r * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    int b = 0;
    while (b < B && !(t >= query_start[b] && t < query_start[b + 1])) ++b;
    if (b == B) { err = -1; continue; }
    int L = query_start[b + 1] - query_start[b];
    int n = context_lens[b];
    if (L > n || n > max_blocks * bs) { err = -1; continue; }
    int npos = n - L + (t - query_start[b]) + 1; /* keys 0 .. npos-1 */
    int g = h / group;
    double* qv = (double*)malloc(sizeof(double) * (size_t)D);
    double* s = (double*)malloc(sizeof(double) * (size_t)npos);
    if (!qv || !s) { free(qv); free(s); err = -2; continue; }
    for (int d = 0; d < D; ++d) qv[d] = load_elem(q, ((size_t)t * Hq + h) * D + d, q_kind);
    int bad = 0;
    for (int i = 0; i < npos; ++i) {
      int blk = block_tables[(size_t)b * max_blocks + i / bs];
      if (blk < 0 || blk >= num_blocks) { bad = 1; break; }
      size_t row = (((size_t)blk * Hkv + g) * bs + i % bs);
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += qv[d] * load_elem(k_cache, row * D + d, cache_kind);
      s[i] = scale * acc;
    }
    if (bad) { err = -1; free(qv); free(s); continue; }
    double m = s[0];
    for (int i = 1; i < npos; ++i) if (s[i] > m) m = s[i];
    double sum = 0.0;
    for (int i = 0; i < npos; ++i) { s[i] = exp(s[i] - m); sum += s[i]; }
    for (int i = 0; i < npos; ++i) s[i] /= sum;
    for (int i = 0; i < npos; ++i) {
      int blk = block_tables[(size_t)b * max_blocks + i / bs];
      size_t row = (((size_t)blk * Hkv + g) * bs + i % bs);
      for (int d = 0; d < D; ++d) o[d] += s[i] * load_elem(v_cache, row * D + d, cache_kind);
    }
    free(qv);
    free(s);
  }
  return err;
}
