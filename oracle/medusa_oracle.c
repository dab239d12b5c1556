/*
 * medusa_oracle.c -- plain CPU oracle for the Medusa tree-verification step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file: it is used by the tests, by the `cpu_baseline` leg of the
 * benchmark and by the smoke check, and by nothing else.  It shares no source
 * with the CUDA library (no headers, tables, helpers or constants).
 *
 * It is written to be read, not to be fast: float64 arithmetic wherever the
 * pages leave the precision open, one loop per definition, no blocking, no
 * fusion.  The only concession to speed is an OpenMP loop over independent
 * (sequence, head, node) outputs.
 *
 * What it follows (the pages state the problem, not formulas):
 *  - vLLM issue 1171 "[Discussion] Will vLLM consider using Speculative
 *    Sampling to accelerating LLM decoding?": several new tokens attend to an
 *    existing paged KV cache (comment by zhaoyang-star), the Medusa tree mask
 *    is applied inside the cached-KV attention, block tables are updated on
 *    acceptance and the other blocks released, and a list of tokens comes back
 *    (comment by void-main listing the needed changes).
 *  - TensorRT-LLM issue 1946 "How to use Medusa to support non llama models?",
 *    answer by rakib-hasan: a position-offset tensor makes RoPE rotate each
 *    Medusa token at its own position (prefix length + tree depth here).
 *  - lmdeploy PR 1231 "[WIP] support Medusa": greedy acceptance at LM-head
 *    temperature 0 (`evaluate_posterior`), verified with a 64-choice tree.
 *  - vLLM issue 1171, opening comment (gesanqiu): a "typical acceptance
 *    scheme" is named beside tree attention but not defined (the reading taken
 *    is stated at or_accept_typical).
 *
 * Readings the pages leave open (the node-0 root at position prefix_len,
 * self-visibility, NeoX half-split RoPE pairing, 1/sqrt(D) scale, lowest index
 * on argmax ties, deepest-then-lowest-index path end, ascending-depth commit,
 * release of scratch pages past the new length, the FP8 E4M3 element format of
 * an FP8 KV cache) are stated at each function.
 *
 * Parity pins: every function here is checked by tests that do not re-type its
 * formula (dense-mask brute force, closed forms, invariants, exhaustive
 * enumeration, hand-derived fixtures, a library's own conversion).  No function
 * is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_F32 = 0, OR_F16 = 1, OR_BF16 = 2, OR_E4M3 = 3 /* FP8 cache element */ };
enum { OR_OK = 0, OR_ERR_ARG = -1, OR_ERR_TREE = -3, OR_ERR_PAGES = -4 };

/* ------------------------------------------------------------------------- */
/* Number formats, written out from the IEEE binary16 and bfloat16 layouts.   */
/* ------------------------------------------------------------------------- */

static double f16_bits_to_double(uint16_t h) {
  int sign = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
  double v;
  if (e == 0) v = ldexp((double)m, -24);               /* zero or subnormal */
  else if (e == 31) v = m ? NAN : INFINITY;
  else v = ldexp((double)(m | 0x400), e - 25);          /* 1.m * 2^(e-15)    */
  return sign ? -v : v;
}

static double bf16_bits_to_double(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Round a finite double to the grid of a binary format with `mant` stored
 * mantissa bits and minimum normal exponent `emin`, ties to even.  Returns the
 * rounded value (exact in double) or +-inf past the largest finite value. */
static double round_to_format(double v, int mant, int emin, double max_finite) {
  double a = fabs(v);
  if (a == 0.0) return v;
  int e;
  frexp(a, &e);                      /* a = m * 2^e, m in [0.5, 1) */
  int E = e - 1;                     /* a in [2^E, 2^(E+1))        */
  if (E < emin) E = emin;            /* subnormals share the smallest quantum */
  double q = ldexp(1.0, E - mant);   /* spacing of representable values */
  double r = nearbyint(a / q) * q;   /* default rounding mode: ties to even */
  if (r > max_finite) r = INFINITY;
  return v < 0 ? -r : r;
}

static uint16_t encode_binary16_like(double r, int mant, int emin, int bias, int expbits) {
  uint16_t s = signbit(r) ? (uint16_t)(1u << 15) : 0;
  double a = fabs(r);
  if (a == 0.0) return s;
  if (isinf(a)) return (uint16_t)(s | (((1u << expbits) - 1u) << mant));
  int e;
  frexp(a, &e);
  int E = e - 1;
  if (E < emin) { /* subnormal: integer multiple of the smallest quantum */
    return (uint16_t)(s | (uint16_t)(a / ldexp(1.0, emin - mant)));
  }
  uint32_t frac = (uint32_t)((a / ldexp(1.0, E) - 1.0) * ldexp(1.0, mant));
  return (uint16_t)(s | ((uint32_t)(E + bias) << mant) | frac);
}

static uint16_t float_to_f16_bits(float f) {
  /* binary16: 10 mantissa bits, emin -14, bias 15, largest finite 65504 */
  double r = round_to_format((double)f, 10, -14, 65504.0);
  return encode_binary16_like(r, 10, -14, 15, 5);
}

static uint16_t float_to_bf16_bits(float f) {
  /* bfloat16: 7 mantissa bits, emin -126, bias 127, largest (2-2^-7)*2^127 */
  double r = round_to_format((double)f, 7, -126, ldexp(255.0, 120));
  return encode_binary16_like(r, 7, -126, 127, 8);
}

static size_t elem_size(int dt) { return dt == OR_F32 ? 4 : dt == OR_E4M3 ? 1 : 2; }

static double load_act(int dt, const void* base, size_t i) {
  if (dt == OR_F32) return (double)((const float*)base)[i];
  uint16_t h = ((const uint16_t*)base)[i];
  return dt == OR_F16 ? f16_bits_to_double(h) : bf16_bits_to_double(h);
}

static void store_act_from_float(int dt, void* base, size_t i, float v) {
  if (dt == OR_F32) ((float*)base)[i] = v;
  else if (dt == OR_F16) ((uint16_t*)base)[i] = float_to_f16_bits(v);
  else ((uint16_t*)base)[i] = float_to_bf16_bits(v);
}

/* Exposed for the tests: round float32 values to fp16 / bf16 bit patterns. */
void or_round_to_act(int dt, long n, const float* x, void* y) {
  for (long i = 0; i < n; ++i) store_act_from_float(dt, y, (size_t)i, x[i]);
}

/* Exposed for the tests: decode act-dtype values to float64. */
void or_act_to_double(int dt, long n, const void* x, double* y) {
  for (long i = 0; i < n; ++i) y[i] = load_act(dt, x, (size_t)i);
}

/* ------------------------------------------------------------------------- */
/* FP8 E4M3 (OCP 8-bit floating point, the variant without infinities), the  */
/* element format of an FP8 KV cache.  Reading (the pages define no FP8      */
/* cache): bits S EEEE MMM, exponent bias 7; E = 0 is subnormal,             */
/* (-1)^S 2^-6 M/8; otherwise (-1)^S 2^(E-7) (1 + M/8); S 1111 111 is NaN,   */
/* so the largest finite magnitude is 2^8 * 1.75 = 448.  Encoding rounds to  */
/* the nearest representable value, ties to the even code (mantissa LSB 0),  */
/* and saturates finite overflow and infinities to +-448; NaN stays NaN.     */
/* ------------------------------------------------------------------------- */

static double e4m3_magnitude(int code7) {  /* code7 = E:M, 0 .. 0x7E */
  int E = code7 >> 3, M = code7 & 7;
  return E == 0 ? ldexp((double)M / 8.0, -6) : ldexp(1.0 + (double)M / 8.0, E - 7);
}

double or_e4m3_decode(int code) {
  int sign = (code >> 7) & 1, mag = code & 0x7F;
  if (mag == 0x7F) return NAN;
  double v = e4m3_magnitude(mag);
  return sign ? -v : v;
}

int or_e4m3_encode(double x) {
  if (isnan(x)) return 0x7F;
  int sign = signbit(x) ? 0x80 : 0;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  /* the nearest of the 127 finite magnitudes; on a tie the even code */
  int best = 0;
  double best_d = a;
  for (int c = 1; c <= 0x7E; ++c) {
    double d = fabs(e4m3_magnitude(c) - a);
    if (d < best_d || (d == best_d && (c & 1) == 0)) {
      best = c;
      best_d = d;
    }
  }
  return sign | best;
}

/* Exposed for the tests: arrays of codes and values. */
void or_e4m3_encode_array(long n, const double* x, uint8_t* codes) {
  for (long i = 0; i < n; ++i) codes[i] = (uint8_t)or_e4m3_encode(x[i]);
}
void or_e4m3_decode_array(long n, const uint8_t* codes, double* x) {
  for (long i = 0; i < n; ++i) x[i] = or_e4m3_decode(codes[i]);
}

int or_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------------- */
/* RoPE with the Medusa position offset.                                      */
/* ------------------------------------------------------------------------- */

/* cos/sin table, [max_pos][D/2] each, fp32.  Definition (NeoX/LLaMA form):
 *   inv_freq_j = pow(base, -(2j)/D)   (IEEE double)
 *   theta      = pos * inv_freq_j     (double multiply)
 *   table      = cos(theta), sin(theta) in double, rounded to fp32. */
void or_rope_table(double base, int head_dim, int max_pos, float* cos_tab, float* sin_tab) {
  int half = head_dim / 2;
  for (int pos = 0; pos < max_pos; ++pos) {
    for (int j = 0; j < half; ++j) {
      double inv_freq = pow(base, -(2.0 * (double)j) / (double)head_dim);
      double theta = (double)pos * inv_freq;
      cos_tab[(size_t)pos * half + j] = (float)cos(theta);
      sin_tab[(size_t)pos * half + j] = (float)sin(theta);
    }
  }
}

/* Rotate n_rows rows of D values, row r at position pos[r] (prefix_len +
 * depth for a tree token; TensorRT-LLM issue 1946, answer on position
 * offsets).  Half-split pairing: element j pairs with j + D/2.  Arithmetic in
 * fp32 exactly as written (no fused multiply-add: build with
 * -ffp-contract=off), then one round-to-nearest-even to the act dtype:
 *   x'[j]       = x[j]*c - x[j+D/2]*s
 *   x'[j+D/2]   = x[j+D/2]*c + x[j]*s                                        */
int or_rope_rotate(int dt, long n_rows, int head_dim, const void* x, const int32_t* pos,
                   int max_pos, const float* cos_tab, const float* sin_tab, void* y) {
  int half = head_dim / 2;
  for (long r = 0; r < n_rows; ++r) {
    if (pos[r] < 0 || pos[r] >= max_pos) return OR_ERR_ARG;
    const float* c_row = cos_tab + (size_t)pos[r] * half;
    const float* s_row = sin_tab + (size_t)pos[r] * half;
    size_t base = (size_t)r * head_dim;
    for (int j = 0; j < half; ++j) {
      float lo = (float)load_act(dt, x, base + j);
      float hi = (float)load_act(dt, x, base + j + half);
      float c = c_row[j], s = s_row[j];
      float a1 = lo * c;
      float a2 = hi * s;
      float out_lo = a1 - a2;
      float b1 = hi * c;
      float b2 = lo * s;
      float out_hi = b1 + b2;
      store_act_from_float(dt, y, base + j, out_lo);
      store_act_from_float(dt, y, base + j + half, out_hi);
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Tree checks.                                                               */
/* ------------------------------------------------------------------------- */

/* A tree of T nodes in topological order: node 0 is the root (parent -1,
 * depth 0) and every other node has 0 <= parent < its own index and depth one
 * more than its parent's. */
static int check_tree(int T, const int32_t* parents, const int32_t* depths) {
  if (T < 1) return OR_ERR_TREE;
  if (parents[0] != -1) return OR_ERR_TREE;
  if (depths && depths[0] != 0) return OR_ERR_TREE;
  for (int i = 1; i < T; ++i) {
    if (parents[i] < 0 || parents[i] >= i) return OR_ERR_TREE;
    if (depths && depths[i] != depths[parents[i]] + 1) return OR_ERR_TREE;
  }
  return OR_OK;
}

int or_check_tree(int T, const int32_t* parents, const int32_t* depths) {
  return check_tree(T, parents, depths);
}

/* ------------------------------------------------------------------------- */
/* Tree attention over the paged prefix.                                      */
/* ------------------------------------------------------------------------- */

/* Address of logical slot `slot` of sequence b, KV head kvh, in a cache laid
 * out as [num_pages][Hkv][P][D]: page = block_tables[b][slot / P], row slot % P.
 * Returns the element offset of the row, or -1 if the table does not cover it. */
static long slot_offset(const int32_t* block_tables, int max_blocks, int num_pages, int Hkv,
                        int P, int D, int b, int kvh, long slot) {
  long blk = slot / P;
  if (blk >= max_blocks) return -1;
  int page = block_tables[(size_t)b * max_blocks + blk];
  if (page < 0 || page >= num_pages) return -1;
  return (((long)page * Hkv + kvh) * P + slot % P) * (long)D;
}

/* For each selected (b, h, i): node i of sequence b, query head h, attends to
 *   - every prefix key, logical slots 0 .. seq_lens[b]-1 of the paged cache,
 *   - the tree keys of its own ancestors, itself included (the Medusa tree
 *     mask; a node sees exactly its root-to-node path),
 * with KV head kvh = h / (Hq/Hkv).  In float64 from the act-dtype inputs:
 *   s_j = (q . k_j) * sm_scale,  p_j = exp(s_j - max s),  o = sum p_j v_j / sum p_j.
 * q_rot and k_rot are already rotated (see or_rope_rotate); the prefix keys in
 * the cache are taken as stored.  out is [n_sel][D] float64. */
int or_tree_attn(int dt, int B, int T, int Hq, int Hkv, int D, int P, int max_blocks,
                 int num_pages, const void* q_rot, const void* k_rot, const void* v_new,
                 const void* k_cache, const void* v_cache, const int32_t* block_tables,
                 const int32_t* seq_lens, const int32_t* parents, double sm_scale, long n_sel,
                 const int32_t* sel, double* out) {
  if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0) return OR_ERR_ARG;
  int g = Hq / Hkv;
  for (int b = 0; b < B; ++b) {
    int st = check_tree(T, parents + (size_t)b * T, NULL);
    if (st) return st;
  }
  int status = OR_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (long n = 0; n < n_sel; ++n) {
    int b = sel[3 * n], h = sel[3 * n + 1], i = sel[3 * n + 2];
    int kvh = h / g;
    long L = seq_lens[b];
    const int32_t* par = parents + (size_t)b * T;
    /* the root-to-node path of i, collected by walking parent links */
    int path[64 + 1];
    int np = 0;
    for (int a = i; a >= 0; a = par[a]) {
      if (np > 64) break;
      path[np++] = a;
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)(L + np));
    double* q = (double*)malloc(sizeof(double) * (size_t)D);
    long* koff = (long*)malloc(sizeof(long) * (size_t)(L > 0 ? L : 1));
    for (int d = 0; d < D; ++d) q[d] = load_act(dt, q_rot, (((size_t)b * T + i) * Hq + h) * D + d);
    int bad = 0;
    for (long j = 0; j < L; ++j) {
      koff[j] = slot_offset(block_tables, max_blocks, num_pages, Hkv, P, D, b, kvh, j);
      if (koff[j] < 0) { bad = 1; break; }
    }
    if (bad) {
#pragma omp critical
      status = OR_ERR_PAGES;
    } else {
      double smax = -INFINITY;
      for (long j = 0; j < L; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * load_act(dt, k_cache, (size_t)koff[j] + d);
        s[j] = dot * sm_scale;
        if (s[j] > smax) smax = s[j];
      }
      for (int a = 0; a < np; ++a) {
        size_t row = (((size_t)b * T + path[a]) * Hkv + kvh) * D;
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * load_act(dt, k_rot, row + d);
        s[L + a] = dot * sm_scale;
        if (s[L + a] > smax) smax = s[L + a];
      }
      double denom = 0.0;
      double* o = out + (size_t)n * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (long j = 0; j < L; ++j) {
        double p = exp(s[j] - smax);
        denom += p;
        for (int d = 0; d < D; ++d) o[d] += p * load_act(dt, v_cache, (size_t)koff[j] + d);
      }
      for (int a = 0; a < np; ++a) {
        double p = exp(s[L + a] - smax);
        denom += p;
        size_t row = (((size_t)b * T + path[a]) * Hkv + kvh) * D;
        for (int d = 0; d < D; ++d) o[d] += p * load_act(dt, v_new, row + d);
      }
      for (int d = 0; d < D; ++d) o[d] /= denom;
    }
    free(s);
    free(q);
    free(koff);
  }
  return status;
}

/* Where the call leaves the tree's K/V: node i's rotated key and raw value go
 * to logical slot seq_lens[b] + i of the paged cache (the tree scratch region,
 * which the block table must cover).  Operates in place on the given cache. */
int or_tree_scatter(int dt, int B, int T, int Hkv, int D, int P, int max_blocks, int num_pages,
                    const void* k_rot, const void* v_new, void* k_cache, void* v_cache,
                    const int32_t* block_tables, const int32_t* seq_lens) {
  size_t es = elem_size(dt);
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i < T; ++i) {
      for (int kvh = 0; kvh < Hkv; ++kvh) {
        long off = slot_offset(block_tables, max_blocks, num_pages, Hkv, P, D, b, kvh,
                               (long)seq_lens[b] + i);
        if (off < 0) return OR_ERR_PAGES;
        size_t src = (((size_t)b * T + i) * Hkv + kvh) * D;
        memcpy((char*)k_cache + (size_t)off * es, (const char*)k_rot + src * es, D * es);
        memcpy((char*)v_cache + (size_t)off * es, (const char*)v_new + src * es, D * es);
      }
    }
  }
  return OR_OK;
}

/* ------------------------------------------------------------------------- */
/* Greedy acceptance.                                                         */
/* ------------------------------------------------------------------------- */

/* Per sequence b (LM head at temperature 0, lmdeploy PR 1231; "it uses the
 * argmax result", vLLM issue 1171):
 *   am[i]   = argmax_v logits[b][i][v], the lowest index among equal maxima
 *             (compared exactly; +0 equals -0);
 *   acc[0]  = true (the root token was decided by the previous step);
 *   acc[i]  = acc[parent[i]] and tokens[i] == am[parent[i]];
 *   end     = the accepted node of largest depth, lowest index among equals;
 *   accept_len[b]  = depth[end] (accepted tree tokens besides the root);
 *   accept_path[b] = node ids root..end, then -1 up to max_depth+1 entries;
 *   next_token[b]  = am[end] (the token the target model adds after the path).
 * Logits are fp32/fp16/bf16 [B][T][V]; no NaNs (precondition). */
/* ------------------------------------------------------------------------- */
/* FP8 KV cache (reading; the pages define no FP8 cache): the cache holds    */
/* E4M3 codes of value / scale, one scale for all of K and one for all of V; */
/* a cached element stands for decode(code) * scale.                         */
/* ------------------------------------------------------------------------- */

/* Tree K/V into an FP8 cache at logical slots L_b + i: the act-dtype rotated
 * key (raw value) divided by its scale in float32, then encoded. */
int or_tree_scatter_e4m3(int dt, int B, int T, int Hkv, int D, int P, int max_blocks, int num_pages,
                         const void* k_rot, const void* v_new, uint8_t* k_cache, uint8_t* v_cache,
                         const int32_t* block_tables, const int32_t* seq_lens, float k_scale,
                         float v_scale) {
  if (!(k_scale > 0.0f) || !(v_scale > 0.0f)) return OR_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    for (int i = 0; i < T; ++i) {
      for (int kvh = 0; kvh < Hkv; ++kvh) {
        long off = slot_offset(block_tables, max_blocks, num_pages, Hkv, P, D, b, kvh,
                               (long)seq_lens[b] + i);
        if (off < 0) return OR_ERR_PAGES;
        size_t src = (((size_t)b * T + i) * Hkv + kvh) * D;
        for (int d = 0; d < D; ++d) {
          float xk = (float)load_act(dt, k_rot, src + d);
          float xv = (float)load_act(dt, v_new, src + d);
          k_cache[(size_t)off + d] = (uint8_t)or_e4m3_encode((double)(xk / k_scale));
          v_cache[(size_t)off + d] = (uint8_t)or_e4m3_encode((double)(xv / v_scale));
        }
      }
    }
  }
  return OR_OK;
}

/* Tree attention over an FP8 cache: node i of sequence b sees the prefix
 * slots [0, L_b) and the tree slots L_b + t of its own root path, every one
 * read from the cache (so the tree's keys and values too are the encoded
 * ones); softmax(q . k * sm_scale) v in float64 with k, v = decode * scale.
 * q_rot is the act-dtype rotated query.  Same selection and output layout as
 * or_tree_attn. */
int or_tree_attn_e4m3(int dt, int B, int T, int Hq, int Hkv, int D, int P, int max_blocks,
                      int num_pages, const void* q_rot, const uint8_t* k_cache,
                      const uint8_t* v_cache, double k_scale, double v_scale,
                      const int32_t* block_tables, const int32_t* seq_lens, const int32_t* parents,
                      double sm_scale, long n_sel, const int32_t* sel, double* out) {
  if (Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || P <= 0) return OR_ERR_ARG;
  int g = Hq / Hkv;
  for (int b = 0; b < B; ++b) {
    int st = check_tree(T, parents + (size_t)b * T, NULL);
    if (st) return st;
  }
  int status = OR_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (long n = 0; n < n_sel; ++n) {
    int b = sel[3 * n], h = sel[3 * n + 1], i = sel[3 * n + 2];
    int kvh = h / g;
    long L = seq_lens[b];
    const int32_t* par = parents + (size_t)b * T;
    /* the visible slots: the prefix, then the root-to-node path of i */
    long nvis = L;
    long* slot = (long*)malloc(sizeof(long) * (size_t)(L + 65));
    for (long j = 0; j < L; ++j) slot[j] = j;
    for (int a = i; a >= 0 && nvis < L + 65; a = par[a]) slot[nvis++] = L + a;
    long* koff = (long*)malloc(sizeof(long) * (size_t)nvis);
    double* s = (double*)malloc(sizeof(double) * (size_t)nvis);
    double* q = (double*)malloc(sizeof(double) * (size_t)D);
    for (int d = 0; d < D; ++d) q[d] = load_act(dt, q_rot, (((size_t)b * T + i) * Hq + h) * D + d);
    int bad = 0;
    for (long j = 0; j < nvis; ++j) {
      koff[j] = slot_offset(block_tables, max_blocks, num_pages, Hkv, P, D, b, kvh, slot[j]);
      if (koff[j] < 0) bad = 1;
    }
    if (bad) {
#pragma omp critical
      status = OR_ERR_PAGES;
    } else {
      double smax = -INFINITY;
      for (long j = 0; j < nvis; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d) dot += q[d] * (or_e4m3_decode(k_cache[(size_t)koff[j] + d]) * k_scale);
        s[j] = dot * sm_scale;
        if (s[j] > smax) smax = s[j];
      }
      double denom = 0.0;
      double* o = out + (size_t)n * D;
      for (int d = 0; d < D; ++d) o[d] = 0.0;
      for (long j = 0; j < nvis; ++j) {
        double p = exp(s[j] - smax);
        denom += p;
        for (int d = 0; d < D; ++d) o[d] += p * (or_e4m3_decode(v_cache[(size_t)koff[j] + d]) * v_scale);
      }
      for (int d = 0; d < D; ++d) o[d] /= denom;
    }
    free(slot);
    free(koff);
    free(s);
    free(q);
  }
  return status;
}

int or_accept_greedy(int dt, int B, int T, int V, int max_depth, const int32_t* tokens,
                     const void* logits, const int32_t* parents, int32_t* argmax_out,
                     int32_t* accept_len, int32_t* accept_path, int32_t* next_token) {
  if (B < 0 || T < 1 || T > 64 || V < 1 || max_depth < 0) return OR_ERR_ARG;
  int status = OR_OK;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parents + (size_t)b * T;
    if (check_tree(T, par, NULL)) { status = OR_ERR_TREE; continue; }
    int depth[64];
    depth[0] = 0;
    for (int i = 1; i < T; ++i) depth[i] = depth[par[i]] + 1;
    int too_deep = 0;
    for (int i = 0; i < T; ++i) if (depth[i] > max_depth) too_deep = 1;
    if (too_deep) { status = OR_ERR_TREE; continue; }
    int am[64];
    for (int i = 0; i < T; ++i) {
      size_t row = ((size_t)b * T + i) * (size_t)V;
      double best = load_act(dt, logits, row);
      int best_v = 0;
      for (int v = 1; v < V; ++v) {
        double x = load_act(dt, logits, row + v);
        if (x > best) { best = x; best_v = v; }
      }
      am[i] = best_v;
      argmax_out[(size_t)b * T + i] = best_v;
    }
    int acc[64];
    acc[0] = 1;
    for (int i = 1; i < T; ++i)
      acc[i] = acc[par[i]] && tokens[(size_t)b * T + i] == am[par[i]];
    int end = 0;
    for (int i = 1; i < T; ++i)
      if (acc[i] && depth[i] > depth[end]) end = i;   /* strict: lowest index wins ties */
    accept_len[b] = depth[end];
    int32_t* path = accept_path + (size_t)b * (max_depth + 1);
    for (int d = 0; d <= max_depth; ++d) path[d] = -1;
    for (int a = end; a >= 0; a = par[a]) path[depth[a]] = a;
    next_token[b] = am[end];
  }
  return status;
}

/* Typical acceptance.  The pages name a "typical acceptance scheme" beside
 * tree attention as the part of Medusa that inference frameworks lack
 * (vLLM issue 1171, opening comment by gesanqiu) but never define it.
 * Reading taken, from the Medusa paper's typical-acceptance rule (Cai et al.,
 * "Medusa: Simple LLM Inference Acceleration Framework with Multiple Decoding
 * Heads", 2024), restated: a tree node i > 0 passes when the target model's
 * tempered distribution at its parent,
 *     q_v = exp(x_v / tau) / sum_u exp(x_u / tau)   (x = the parent's logits row),
 * gives its token more than
 *     thr = min(epsilon, delta * exp(-H)),   H = -sum_v q_v ln q_v   (nats),
 * i.e. q[token_i] > thr (a token outside [0, V) has q = 0 and fails).  The
 * root always passes.  The accepted path is then chosen exactly as in greedy
 * acceptance (every node on the root path passes; deepest end, lowest index
 * among equals), and next_token is the end row's argmax (the bonus token at
 * temperature 0: no random draw).
 * Outputs per node: node_accept (the node's own test, 1 at the root),
 * prob = q[token_i] and thr of its parent's row (1 and 0 at the root). */
int or_accept_typical(int dt, int B, int T, int V, int max_depth, const int32_t* tokens,
                      const void* logits, const int32_t* parents, double tau, double epsilon,
                      double delta, int32_t* node_accept, double* prob, double* thr,
                      int32_t* accept_len, int32_t* accept_path, int32_t* next_token) {
  if (B < 0 || T < 1 || T > 64 || V < 1 || max_depth < 0) return OR_ERR_ARG;
  if (!(tau > 0.0) || !(epsilon > 0.0) || !(delta > 0.0) || isinf(tau) || isinf(epsilon) ||
      isinf(delta))
    return OR_ERR_ARG;
  int status = OR_OK;
  double* q = (double*)malloc(sizeof(double) * (size_t)V);
  if (!q) return OR_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parents + (size_t)b * T;
    const int32_t* tok = tokens + (size_t)b * T;
    if (check_tree(T, par, NULL)) { status = OR_ERR_TREE; continue; }
    int depth[64];
    depth[0] = 0;
    for (int i = 1; i < T; ++i) depth[i] = depth[par[i]] + 1;
    int too_deep = 0;
    for (int i = 0; i < T; ++i) if (depth[i] > max_depth) too_deep = 1;
    if (too_deep) { status = OR_ERR_TREE; continue; }
    /* each node's own test, under its parent's tempered distribution */
    int pass[64];
    pass[0] = 1;
    node_accept[(size_t)b * T] = 1;
    prob[(size_t)b * T] = 1.0;
    thr[(size_t)b * T] = 0.0;
    for (int i = 1; i < T; ++i) {
      const size_t row = ((size_t)b * T + par[i]) * (size_t)V;
      double m = -INFINITY;
      for (int v = 0; v < V; ++v) {
        const double xv = load_act(dt, logits, row + v) / tau;
        if (xv > m) m = xv;
      }
      double z = 0.0;
      for (int v = 0; v < V; ++v) {
        q[v] = exp(load_act(dt, logits, row + v) / tau - m);
        z += q[v];
      }
      double h = 0.0;
      for (int v = 0; v < V; ++v) {
        q[v] /= z;
        if (q[v] > 0.0) h -= q[v] * log(q[v]);
      }
      const double t = fmin(epsilon, delta * exp(-h));
      const double pt = (tok[i] >= 0 && tok[i] < V) ? q[tok[i]] : 0.0;
      pass[i] = pt > t;
      node_accept[(size_t)b * T + i] = pass[i];
      prob[(size_t)b * T + i] = pt;
      thr[(size_t)b * T + i] = t;
    }
    int acc[64];
    acc[0] = 1;
    for (int i = 1; i < T; ++i) acc[i] = acc[par[i]] && pass[i];
    int end = 0;
    for (int i = 1; i < T; ++i)
      if (acc[i] && depth[i] > depth[end]) end = i;   /* strict: lowest index wins ties */
    accept_len[b] = depth[end];
    int32_t* path = accept_path + (size_t)b * (max_depth + 1);
    for (int d = 0; d <= max_depth; ++d) path[d] = -1;
    for (int a = end; a >= 0; a = par[a]) path[depth[a]] = a;
    const size_t erow = ((size_t)b * T + end) * (size_t)V;
    double best = load_act(dt, logits, erow);
    int best_v = 0;
    for (int v = 1; v < V; ++v) {
      const double x = load_act(dt, logits, erow + v);
      if (x > best) { best = x; best_v = v; }
    }
    next_token[b] = best_v;
  }
  free(q);
  return status;
}

/* ------------------------------------------------------------------------- */
/* KV commit.                                                                 */
/* ------------------------------------------------------------------------- */

/* Keep the accepted nodes' K/V and release the rest (vLLM issue 1171,
 * void-main: "update block tables when you accept one candidate and release
 * other blocks").  For each sequence b with L = accept_len[b], len = seq_lens[b]:
 *   for d = 0..L, ascending: every KV head's K and V row at logical slot
 *     len + accept_path[b][d] is copied to slot len + d (all of one sequence's
 *     sources are read before any of its destinations is written);
 *   seq_lens[b] = len + L + 1;
 *   every logical block p with p*P >= len + L + 1 that holds tree scratch
 *     (p*P < len + T) is released: its page id goes, in ascending p, to
 *     released_pages[b][*] (padded with -1, width rel_width) and
 *     block_tables[b][p] becomes -1.
 * Operates in place on caller-supplied copies. */
int or_kv_commit(int dt, int B, int T, int Hkv, int D, int P, int max_blocks, int num_pages,
                 int max_depth, const int32_t* accept_path, const int32_t* accept_len,
                 void* k_cache, void* v_cache, int32_t* block_tables, int32_t* seq_lens,
                 int32_t* released_pages, int rel_width) {
  size_t es = elem_size(dt);
  size_t row_bytes = (size_t)D * es;
  int status = OR_OK;
  for (int b = 0; b < B; ++b) {
    long len = seq_lens[b];
    int L = accept_len[b];
    const int32_t* path = accept_path + (size_t)b * (max_depth + 1);
    int32_t* rel = released_pages + (size_t)b * rel_width;
    for (int r = 0; r < rel_width; ++r) rel[r] = -1;
    if (L < 0 || L > max_depth || L >= T) { status = OR_ERR_ARG; continue; }
    int ok = 1;
    for (int d = 0; d <= L; ++d) if (path[d] < 0 || path[d] >= T) ok = 0;
    if (!ok) { status = OR_ERR_ARG; continue; }
    /* gather all sources first */
    char* kbuf = (char*)malloc(row_bytes * (size_t)(L + 1) * Hkv);
    char* vbuf = (char*)malloc(row_bytes * (size_t)(L + 1) * Hkv);
    for (int d = 0; d <= L && ok; ++d) {
      for (int kvh = 0; kvh < Hkv; ++kvh) {
        long src = slot_offset(block_tables, max_blocks, num_pages, Hkv, P, D, b, kvh,
                               len + path[d]);
        if (src < 0) { ok = 0; break; }
        memcpy(kbuf + ((size_t)d * Hkv + kvh) * row_bytes, (char*)k_cache + (size_t)src * es, row_bytes);
        memcpy(vbuf + ((size_t)d * Hkv + kvh) * row_bytes, (char*)v_cache + (size_t)src * es, row_bytes);
      }
    }
    for (int d = 0; d <= L && ok; ++d) {
      for (int kvh = 0; kvh < Hkv; ++kvh) {
        long dst = slot_offset(block_tables, max_blocks, num_pages, Hkv, P, D, b, kvh, len + d);
        if (dst < 0) { ok = 0; break; }
        memcpy((char*)k_cache + (size_t)dst * es, kbuf + ((size_t)d * Hkv + kvh) * row_bytes, row_bytes);
        memcpy((char*)v_cache + (size_t)dst * es, vbuf + ((size_t)d * Hkv + kvh) * row_bytes, row_bytes);
      }
    }
    free(kbuf);
    free(vbuf);
    if (!ok) { status = OR_ERR_PAGES; continue; }
    long new_len = len + L + 1;
    seq_lens[b] = (int32_t)new_len;
    int nrel = 0;
    for (long p = 0; p < max_blocks; ++p) {
      if (p * P >= new_len && p * P < len + T) {
        int32_t* entry = block_tables + (size_t)b * max_blocks + p;
        if (nrel < rel_width) rel[nrel++] = *entry;
        *entry = -1;
      }
    }
  }
  return status;
}

/* ------------------------------------------------------------------------- */
/* Candidate tree tokens from the base and Medusa-head logits                 */
/* (lmdeploy PR 1231 "[WIP] support Medusa": generate_candidates; Medusa heads */
/* at top-k over a 64-choice tree).  Reading: node 0 takes the argmax of the   */
/* base logits; a node at depth d with r earlier siblings takes the entry of   */
/* rank r of head d-1, ranked by larger value first, lower index first among   */
/* equal values.  The entry of rank r is found by r+1 successive selections,   */
/* each of the best entry ranked after the previous one.                      */
/* ------------------------------------------------------------------------- */

/* 1 if (v, i) ranks before (w, j). */
static int ranks_before(double v, int i, double w, int j) {
  return v > w || (v == w && i < j);
}

static int rank_entry(int dt, const void* logits, size_t row, int V, int r) {
  double pv = 0.0;
  int pi = -1;  /* previous selection; none yet */
  for (int k = 0; k <= r; ++k) {
    double bv = 0.0;
    int bi = -1;
    for (int v = 0; v < V; ++v) {
      double x = load_act(dt, logits, row + v);
      if (pi >= 0 && !ranks_before(pv, pi, x, v)) continue; /* not after the previous one */
      if (bi < 0 || ranks_before(x, v, bv, bi)) { bv = x; bi = v; }
    }
    if (bi < 0) return -1; /* fewer than r+1 entries */
    pv = bv;
    pi = bi;
  }
  return pi;
}

int or_tree_candidates(int dt, int B, int T, int heads, int V, const void* root_logits,
                       const void* head_logits, const int32_t* parents, int32_t* tokens) {
  if (B < 0 || T < 1 || T > 64 || heads < 1 || V < 1) return OR_ERR_ARG;
  int status = OR_OK;
  for (int b = 0; b < B; ++b) {
    const int32_t* par = parents + (size_t)b * T;
    if (check_tree(T, par, NULL)) { status = OR_ERR_TREE; continue; }
    int depth[64];
    depth[0] = 0;
    for (int i = 1; i < T; ++i) depth[i] = depth[par[i]] + 1;
    int bad = 0;
    for (int i = 0; i < T; ++i) if (depth[i] > heads) bad = 1;
    if (bad) { status = OR_ERR_TREE; continue; }
    tokens[(size_t)b * T] = rank_entry(dt, root_logits, (size_t)b * V, V, 0);
    for (int i = 1; i < T; ++i) {
      int r = 0;
      for (int j = 1; j < i; ++j) if (par[j] == par[i]) ++r;
      size_t row = ((size_t)b * heads + (depth[i] - 1)) * (size_t)V;
      tokens[(size_t)b * T + i] = rank_entry(dt, head_logits, row, V, r);
    }
  }
  return status;
}
