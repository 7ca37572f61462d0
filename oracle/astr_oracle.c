/*
 * astr_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow CPU definition of the paged KV-cache attention path: RoPE applied to Q/K from
 * an f32 [cos, sin] table and written into the cache at out_cache_loc, then GQA
 * softmax(q.k/sqrt(d)).v over the paged cache for decode (optionally split into chunks merged
 * by log-sum-exp) and for varlen causal prefill; on the training path, RoPE with no cache
 * write and its backward (the rotation by -theta). Attention is evaluated in double precision
 * from the stored (f32 or bf16) values; nothing is blocked, fused or reordered beyond the
 * definitions cited at each function.
 *
 * Only the tests, __graft_entry__.smoke() and bench.py's CPU-baseline leg may load this
 * library. It shares no code, header or table with the CUDA library. Build:
 *   gcc -O2 -std=c11 -ffp-contract=off -fopenmp -fPIC -shared astr_oracle.c -o liboracle.so -lm
 * (-ffp-contract=off keeps every float product and sum separately rounded, which the RoPE
 * rounding specification below relies on.)
 *
 * Sources (the AstrAI documentation pages):
 *   [INT-MASK]  AstrAI internals, "Autoregression & Causal Masking": the lower-triangular
 *               0 / -inf mask; position i attends to positions <= i.
 *   [INT-ROPE]  AstrAI internals, "Rotary Position Embedding (RoPE)": q_i = R_i W_q x_i,
 *               freqs_cis [max_len, dim/2, 2] f32 [cos, sin]; RoPE before the cache write.
 *   [INT-KV]    AstrAI internals, "KV Cache Mathematics": o_n = sum_j softmax(q_n k_j/sqrt(d_k)) v_j.
 *   [INT-BE]    AstrAI internals, "Attention Backend": blhd layout, scale always 1/sqrt(head_dim).
 *   [INF-KVC]   AstrAI inference guide, "KVCache System": KVCache fields, raw indexing
 *               k_buffer[layer_id, out_cache_loc] = k, decode_o_part / decode_ml_part merge.
 *   [INF-ROT]   AstrAI inference guide, "Rotary Embedding Backend": the torch path multiplies
 *               view_as_complex pairs, i.e. adjacent elements (x[2i], x[2i+1]).
 *   [INF-BE]    AstrAI inference guide, "Attention Backend": paged decode through req_to_token;
 *               ragged prefill through qo_indptr + kv_indptr.
 *   [INF-RADIX] AstrAI inference guide, "KVCache System": prefill resumes right after the
 *               longest complete-page prefix hit.
 *   [PAPER-GQA] AstrAI paper, "Model Architecture": GQA with shared KV heads.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   R1  GQA: query head h reads KV head floor(h / (n_heads / n_kv_heads)).
 *   R2  Decode: the query of request b sits at position seq_lens[b]-1 and attends all
 *       seq_lens[b] cached positions, its own freshly written token included.
 *   R3  Prefill: row i of request b has absolute position P_b + i, P_b = kv_len - q_len, and
 *       attends keys 0..P_b+i (the mask is aligned to absolute positions).
 *   R4  Split-K: decode_o_part gains a split axis [B, H, S, D] holding normalised partial
 *       outputs; decode_ml_part holds (m_s, l_s) per split in natural-exponent units.
 *   R5  RoPE rounding: the rotation is evaluated in f32 with every product and sum rounded
 *       separately (no fused multiply-add): a' = RN(RN(a c) - RN(b s)),
 *       b' = RN(RN(a s) + RN(b c)); bf16 inputs are widened exactly and the result is
 *       rounded to bf16 (nearest, ties to even).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_F32 0
#define ORC_BF16 1

/* ------------------------------------------------------------------------------------------ */
/* element access                                                                             */
/* ------------------------------------------------------------------------------------------ */

static float bf16_bits_to_f32(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint16_t f32_to_bf16_bits_rne(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
  uint32_t lsb = (u >> 16) & 1u;
  return (uint16_t)((u + 0x7FFFu + lsb) >> 16);
}

static double load_elem(const void *base, int dtype, int64_t i) {
  if (dtype == ORC_BF16) return (double)bf16_bits_to_f32(((const uint16_t *)base)[i]);
  return (double)((const float *)base)[i];
}

static float load_f32(const void *base, int dtype, int64_t i) {
  if (dtype == ORC_BF16) return bf16_bits_to_f32(((const uint16_t *)base)[i]);
  return ((const float *)base)[i];
}

static void store_f32_as(void *base, int dtype, int64_t i, float v) {
  if (dtype == ORC_BF16)
    ((uint16_t *)base)[i] = f32_to_bf16_bits_rne(v);
  else
    ((float *)base)[i] = v;
}

/* ------------------------------------------------------------------------------------------ */
/* [INT-MASK] causal mask                                                                     */
/* ------------------------------------------------------------------------------------------ */

/* Entry (i, j) of the lower-triangular causal mask: 0 where key j <= query i, else -inf. */
static double causal_mask_entry(int64_t i, int64_t j) { return (j <= i) ? 0.0 : -INFINITY; }

void oracle_causal_mask(int n, double *out) {
  for (int i = 0; i < n; ++i)
    for (int j = 0; j < n; ++j) out[(int64_t)i * n + j] = causal_mask_entry(i, j);
}

/* ------------------------------------------------------------------------------------------ */
/* [INT-ROPE] [INF-ROT] rotary embedding                                                      */
/* ------------------------------------------------------------------------------------------ */

/*
 * Exact rotation in double precision: for each adjacent pair (x[2i], x[2i+1]) read as the
 * complex number a + ib, multiply by the table entry c + is of the row's position:
 *   out[2i] = a c - b s,  out[2i+1] = a s + b c.
 * x: [T, nh, D] doubles; freqs: [max_len, D/2, 2] doubles; pos: [T].
 * Returns the number of tokens whose position falls outside the table (left untouched).
 */
int oracle_rope_f64(int64_t T, int nh, int D, const double *x, const double *freqs,
                    int max_len, const int32_t *pos, double *out) {
  int bad = 0;
  for (int64_t t = 0; t < T; ++t) {
    if (pos[t] < 0 || pos[t] >= max_len) {
      ++bad;
      continue;
    }
    const double *cs = freqs + (int64_t)pos[t] * D;
    for (int h = 0; h < nh; ++h) {
      const double *xr = x + (t * nh + h) * D;
      double *yr = out + (t * nh + h) * D;
      for (int i = 0; i < D / 2; ++i) {
        double a = xr[2 * i], b = xr[2 * i + 1], c = cs[2 * i], s = cs[2 * i + 1];
        yr[2 * i] = a * c - b * s;
        yr[2 * i + 1] = a * s + b * c;
      }
    }
  }
  return bad;
}

/*
 * The same rotation under rounding specification R5 (f32, no fused multiply-add). With
 * `conj` set the table entry is conjugated (c - is): the rotation by -theta, R^T.
 */
static void rotate_row_f32_dir(int dtype, const void *src, int64_t src_off, void *dst,
                               int64_t dst_off, const float *cs, int D, int conj) {
  for (int i = 0; i < D / 2; ++i) {
    float a = load_f32(src, dtype, src_off + 2 * i);
    float b = load_f32(src, dtype, src_off + 2 * i + 1);
    float c = cs[2 * i], s = conj ? -cs[2 * i + 1] : cs[2 * i + 1];
    float ac = a * c, bs = b * s, as = a * s, bc = b * c;
    float re = ac - bs;
    float im = as + bc;
    store_f32_as(dst, dtype, dst_off + 2 * i, re);
    store_f32_as(dst, dtype, dst_off + 2 * i + 1, im);
  }
}

static void rotate_row_f32(int dtype, const void *src, int64_t src_off, void *dst, int64_t dst_off,
                           const float *cs, int D) {
  rotate_row_f32_dir(dtype, src, src_off, dst, dst_off, cs, D, 0);
}

/*
 * RoPE on the training path, with no cache write ([INT-ROPE]: training applies the rotation
 * as a complex multiply that autograd differentiates; [INF-ROT]: the torch complex path).
 * For every token t and head h of x [T, nh, D]:
 *   inverse = 0:  out[t, h] = R_{pos[t]} x[t, h]      (the forward rotation by theta)
 *   inverse = 1:  out[t, h] = R_{pos[t]}^T x[t, h]    (rotation by -theta)
 * The rotation is linear in x with the real 2x2 matrix [[c, -s], [s, c]] per pair, so the
 * gradient of a loss with respect to x is R^T applied to its gradient with respect to out:
 * inverse = 1 is the backward pass (the complex multiply by the conjugate c - is). Both use
 * rounding specification R5. A token whose position falls outside the table is skipped and
 * counted in the return value.
 */
int oracle_rope_apply(int dtype, int64_t T, int nh, int D, const void *x, const float *freqs,
                      int freqs_max_len, const int32_t *pos, int inverse, void *out) {
  int bad = 0;
  for (int64_t t = 0; t < T; ++t) {
    if (pos[t] < 0 || pos[t] >= freqs_max_len) {
      ++bad;
      continue;
    }
    const float *cs = freqs + (int64_t)pos[t] * D;
    for (int h = 0; h < nh; ++h)
      rotate_row_f32_dir(dtype, x, (t * nh + h) * D, out, (t * nh + h) * D, cs, D, inverse);
  }
  return bad;
}

/*
 * Fused step of [INT-ROPE] and [INF-KVC]: for every token t,
 *   q_out[t, h]                     = R_{pos[t]} q[t, h]     (h < H)
 *   k_layer[out_cache_loc[t], g]    = R_{pos[t]} k[t, g]     (g < Hk)
 *   v_layer[out_cache_loc[t], g]    = v[t, g]                (copied unchanged)
 * The rotation happens before the write, so the cached K carries its own position's rotation.
 * k_layer / v_layer point at one layer's [size, Hk, D] slab. A token whose position or slot
 * is out of range is skipped entirely and counted in the return value.
 */
int oracle_rope_kv_write(int dtype, int64_t T, int H, int Hk, int D, const void *q,
                         const void *k, const void *v, const float *freqs, int freqs_max_len,
                         const int32_t *pos, const int32_t *loc, int64_t size, void *q_out,
                         void *k_layer, void *v_layer) {
  int bad = 0;
  for (int64_t t = 0; t < T; ++t) {
    if (pos[t] < 0 || pos[t] >= freqs_max_len || loc[t] < 0 || (int64_t)loc[t] >= size) {
      ++bad;
      continue;
    }
    const float *cs = freqs + (int64_t)pos[t] * D;
    for (int h = 0; h < H; ++h) rotate_row_f32(dtype, q, (t * H + h) * D, q_out, (t * H + h) * D, cs, D);
    int64_t slot = loc[t];
    for (int g = 0; g < Hk; ++g) {
      rotate_row_f32(dtype, k, (t * Hk + g) * D, k_layer, (slot * Hk + g) * D, cs, D);
      for (int e = 0; e < D; ++e) {
        if (dtype == ORC_BF16)
          ((uint16_t *)v_layer)[(slot * Hk + g) * D + e] = ((const uint16_t *)v)[(t * Hk + g) * D + e];
        else
          ((float *)v_layer)[(slot * Hk + g) * D + e] = ((const float *)v)[(t * Hk + g) * D + e];
      }
    }
  }
  return bad;
}

/* ------------------------------------------------------------------------------------------ */
/* attention over a gathered key set                                                          */
/* ------------------------------------------------------------------------------------------ */

/*
 * One query vector against keys j = 0..n_keys-1 of one request's page-table row:
 *   s_j = (q . k_j) / sqrt(D) + mask_j,  w = softmax(s),  o = sum_j w_j v_j      [INT-KV][INT-BE]
 * slot_of_j = row[j] (req_to_token[req_pool_indices[b], j]); KV head g. If qpos >= 0 the
 * causal mask entry (qpos, j) is added ([INT-MASK], reading R3); qpos < 0 means no mask.
 * The softmax is evaluated as exp(s_j - max s) / sum exp(s - max s), the same quotient.
 * Scratch `s` holds n_keys doubles. Returns -1 if a slot is out of range.
 */
static int attend_one(int dtype, int Hk, int D, const void *q, int64_t q_off,
                      const void *k_layer, const void *v_layer, int64_t size,
                      const int32_t *row, int64_t n_keys, int g, int64_t qpos, double *s,
                      double *o) {
  const double scale = 1.0 / sqrt((double)D);
  double m = -INFINITY;
  for (int64_t j = 0; j < n_keys; ++j) {
    int64_t slot = row[j];
    if (slot < 0 || slot >= size) return -1;
    double dot = 0.0;
    for (int e = 0; e < D; ++e)
      dot += load_elem(q, dtype, q_off + e) * load_elem(k_layer, dtype, (slot * Hk + g) * D + e);
    s[j] = dot * scale + (qpos >= 0 ? causal_mask_entry(qpos, j) : 0.0);
    if (s[j] > m) m = s[j];
  }
  double denom = 0.0;
  for (int64_t j = 0; j < n_keys; ++j) {
    s[j] = exp(s[j] - m);
    denom += s[j];
  }
  for (int e = 0; e < D; ++e) o[e] = 0.0;
  for (int64_t j = 0; j < n_keys; ++j) {
    if (s[j] == 0.0) continue;
    int64_t slot = row[j];
    double w = s[j] / denom;
    for (int e = 0; e < D; ++e) o[e] += w * load_elem(v_layer, dtype, (slot * Hk + g) * D + e);
  }
  return 0;
}

/* ------------------------------------------------------------------------------------------ */
/* [INT-KV] [INF-KVC] [INF-BE] decode                                                         */
/* ------------------------------------------------------------------------------------------ */

/*
 * Paged decode: for each selected request b and head h, with L = seq_lens[b] and the
 * request's page-table row req_to_token[req_pool_indices[b]],
 *   out[b, h] = sum_{j<L} softmax_j(q[b,h] . k_{row[j], h/G} / sqrt(D)) v_{row[j], h/G}
 * (readings R1, R2). q: [B, H, D]; out: [B, H, D] doubles. sel (n_sel entries) lists the
 * requests to evaluate; NULL means all B. Returns the number of failed (request, head) units
 * (L < 1, L > max_ctx, bad row or slot).
 */
int oracle_decode(int dtype, int B, int H, int Hk, int D, const void *q, const void *k_layer,
                  const void *v_layer, int64_t size, const int32_t *req_to_token, int num_reqs,
                  int max_ctx, const int32_t *req_pool_indices, const int32_t *seq_lens,
                  int n_sel, const int32_t *sel, double *out) {
  const int G = H / Hk;
  const int nb = sel ? n_sel : B;
  int fails = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : fails)
  for (int64_t u = 0; u < (int64_t)nb * H; ++u) {
    int b = sel ? sel[u / H] : (int)(u / H);
    int h = (int)(u % H);
    int64_t L = seq_lens[b];
    int r = req_pool_indices[b];
    if (L < 1 || L > max_ctx || r < 0 || r >= num_reqs) {
      ++fails;
      continue;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)L);
    if (attend_one(dtype, Hk, D, q, ((int64_t)b * H + h) * D, k_layer, v_layer, size,
                   req_to_token + (int64_t)r * max_ctx, L, h / G, -1, s,
                   out + ((int64_t)b * H + h) * D) != 0)
      ++fails;
    free(s);
  }
  return fails;
}

/*
 * Split-K decode ([INF-KVC] decode_o_part / decode_ml_part, reading R4). For request b the
 * positions are cut into chunks [sC, min((s+1)C, L)), s < ceil(L/C). For each chunk:
 *   m_s = max_j s_j,  l_s = sum_j exp(s_j - m_s),  o_s = sum_j exp(s_j - m_s) v_j / l_s,
 * and the chunks are merged by log-sum-exp:
 *   M = max_s m_s,  w_s = l_s exp(m_s - M),  out = sum_s w_s o_s / sum_s w_s.
 * o_part: [B, H, S, D]; m_part, l_part: [B, H, S]; out: [B, H, D] (all doubles).
 * Entries of splits past ceil(L/C) are left untouched. Returns failed units.
 */
int oracle_decode_split(int dtype, int B, int H, int Hk, int D, const void *q,
                        const void *k_layer, const void *v_layer, int64_t size,
                        const int32_t *req_to_token, int num_reqs, int max_ctx,
                        const int32_t *req_pool_indices, const int32_t *seq_lens, int chunk,
                        int max_splits, double *o_part, double *m_part, double *l_part,
                        double *out) {
  const int G = H / Hk;
  const double scale = 1.0 / sqrt((double)D);
  int fails = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : fails)
  for (int64_t u = 0; u < (int64_t)B * H; ++u) {
    int b = (int)(u / H), h = (int)(u % H), g = h / G;
    int64_t L = seq_lens[b];
    int r = req_pool_indices[b];
    int64_t n_split = (L + chunk - 1) / chunk;
    if (L < 1 || L > max_ctx || r < 0 || r >= num_reqs || chunk < 1 || n_split > max_splits) {
      ++fails;
      continue;
    }
    const int32_t *row = req_to_token + (int64_t)r * max_ctx;
    int64_t qo = ((int64_t)b * H + h) * D;
    double *s = (double *)malloc(sizeof(double) * (size_t)chunk);
    int bad = 0;
    for (int64_t sp = 0; sp < n_split && !bad; ++sp) {
      int64_t j0 = sp * chunk, j1 = (sp + 1) * chunk < L ? (sp + 1) * chunk : L;
      double m = -INFINITY;
      for (int64_t j = j0; j < j1; ++j) {
        int64_t slot = row[j];
        if (slot < 0 || slot >= size) {
          bad = 1;
          break;
        }
        double dot = 0.0;
        for (int e = 0; e < D; ++e)
          dot += load_elem(q, dtype, qo + e) * load_elem(k_layer, dtype, (slot * Hk + g) * D + e);
        s[j - j0] = dot * scale;
        if (s[j - j0] > m) m = s[j - j0];
      }
      if (bad) break;
      double l = 0.0;
      for (int64_t j = j0; j < j1; ++j) {
        s[j - j0] = exp(s[j - j0] - m);
        l += s[j - j0];
      }
      int64_t pidx = ((int64_t)b * H + h) * max_splits + sp;
      double *op = o_part + pidx * D;
      for (int e = 0; e < D; ++e) op[e] = 0.0;
      for (int64_t j = j0; j < j1; ++j) {
        int64_t slot = row[j];
        for (int e = 0; e < D; ++e) op[e] += s[j - j0] * load_elem(v_layer, dtype, (slot * Hk + g) * D + e);
      }
      for (int e = 0; e < D; ++e) op[e] /= l;
      m_part[pidx] = m;
      l_part[pidx] = l;
    }
    free(s);
    if (bad) {
      ++fails;
      continue;
    }
    double M = -INFINITY;
    for (int64_t sp = 0; sp < n_split; ++sp) {
      double ms = m_part[((int64_t)b * H + h) * max_splits + sp];
      if (ms > M) M = ms;
    }
    double wsum = 0.0;
    double *o = out + qo;
    for (int e = 0; e < D; ++e) o[e] = 0.0;
    for (int64_t sp = 0; sp < n_split; ++sp) {
      int64_t pidx = ((int64_t)b * H + h) * max_splits + sp;
      double w = l_part[pidx] * exp(m_part[pidx] - M);
      wsum += w;
      for (int e = 0; e < D; ++e) o[e] += w * o_part[pidx * D + e];
    }
    for (int e = 0; e < D; ++e) o[e] /= wsum;
  }
  return fails;
}

/* ------------------------------------------------------------------------------------------ */
/* [INF-BE] [INF-RADIX] [INT-MASK] varlen causal prefill                                      */
/* ------------------------------------------------------------------------------------------ */

/*
 * Ragged prefill: q is packed by qo_indptr ([sum q, H, D]); request b owns rows
 * qo_indptr[b]..qo_indptr[b+1]-1 and keys 0..K_b-1 of its page-table row, K_b =
 * kv_indptr[b+1]-kv_indptr[b]. Row i of request b has absolute position P_b + i with
 * P_b = K_b - Q_b (reading R3) and
 *   out[t, h] = sum_{j<K_b} softmax_j(q[t,h] . k_{row[j], h/G} / sqrt(D) + mask(P_b+i, j)) v_{row[j], h/G}.
 * rows (n_rows entries) lists the packed rows to evaluate, NULL means all; out is
 * [n_rows, H, D] doubles in the order of `rows`. Returns failed units.
 */
int oracle_prefill(int dtype, int B, int H, int Hk, int D, const void *q, const void *k_layer,
                   const void *v_layer, int64_t size, const int32_t *req_to_token, int num_reqs,
                   int max_ctx, const int32_t *req_pool_indices, const int32_t *qo_indptr,
                   const int32_t *kv_indptr, int64_t n_rows, const int32_t *rows, double *out) {
  const int G = H / Hk;
  const int64_t total = qo_indptr[B];
  const int64_t nr = rows ? n_rows : total;
  int fails = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : fails)
  for (int64_t u = 0; u < nr * H; ++u) {
    int64_t ri = u / H;
    int h = (int)(u % H);
    int64_t t = rows ? rows[ri] : ri;
    if (t < 0 || t >= total) {
      ++fails;
      continue;
    }
    int b = 0;
    while (b + 1 < B && qo_indptr[b + 1] <= t) ++b;
    int64_t Qb = qo_indptr[b + 1] - qo_indptr[b];
    int64_t Kb = (int64_t)kv_indptr[b + 1] - kv_indptr[b];
    int64_t Pb = Kb - Qb;
    int64_t i = t - qo_indptr[b];
    int r = req_pool_indices[b];
    if (Pb < 0 || Kb > max_ctx || r < 0 || r >= num_reqs) {
      ++fails;
      continue;
    }
    double *s = (double *)malloc(sizeof(double) * (size_t)(Kb > 0 ? Kb : 1));
    if (attend_one(dtype, Hk, D, q, (t * H + h) * D, k_layer, v_layer, size,
                   req_to_token + (int64_t)r * max_ctx, Kb, h / G, Pb + i, s,
                   out + (ri * H + h) * D) != 0)
      ++fails;
    free(s);
  }
  return fails;
}

/* Number of OpenMP threads the oracle runs on (1 when built without OpenMP). */
int oracle_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  omp_set_num_threads(n);
#else
  (void)n;
#endif
}
