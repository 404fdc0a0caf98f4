/*
 * mla_oracle.c — plain fp64 CPU oracle for MLA decode over a paged latent
 * KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference legs may load this library.  It shares
 * no code, header, table or constant with the CUDA library; both sides only
 * receive the same seeded inputs.
 *
 * What it computes is the non-absorbed ("decompress") path of the MLA
 * operator write-up (nxmr.cn/news/151634), §4 equivalence script, "path A":
 *   1. widen every bf16 input to double;
 *   2. gather the cache rows of a sequence through its block table (the paged
 *      cache of §3: page_size tokens per page, row = [latent | k_R]);
 *   3. decompress, per head h and token s, K_h[s] = W_UK[h] . c[s] and
 *      V_h[s] = W_UV[h] . c[s] (einsum sc,hdc->shd), with c[s] the latent
 *      slice of the head's group (grouped latent attention, "From MLA to GLA"
 *      §1; G = 1 is plain MLA);
 *   4. score_s = (q_nope . K_h[s] + q_rope . k_R[s]) * scale for the visible
 *      keys s <= n - Lq + l (causal among the Lq new tokens);
 *   5. textbook softmax exp(score - max) / sum, out = sum_s p_s V_h[s],
 *      plus the latent o_lat = sum_s p_s c[s] and lse = max + log(sum).
 * The absorbed score path ("path B", q_abs = q_nope . W_UK) exists here only
 * for the self-check that both paths give the same scores.
 *
 * No blocking, fusion or reordering beyond the definition: plain loops.
 * OpenMP (when compiled with -fopenmp) only distributes independent
 * (sequence, head) pairs over host threads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double bf16_to_double(uint16_t v) {
  uint32_t u = ((uint32_t)v) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * One FP8 code, OCP 8-bit floating point E4M3 ("OFP8" specification): bit 7
 * sign, bits 6..3 exponent with bias 7, bits 2..0 mantissa.  Exponent 0
 * holds the subnormals m/8 * 2^-6; S.1111.111 is NaN; there are no
 * infinities.  Returns the value in double (NaN for the two NaN codes).
 */
double mla_oracle_e4m3(int code) {
  const int s = (code >> 7) & 1, e = (code >> 3) & 15, m = code & 7;
  if (e == 15 && m == 7) return NAN;
  const double v = e == 0 ? ldexp((double)m / 8.0, -6) : ldexp(1.0 + (double)m / 8.0, e - 7);
  return s ? -v : v;
}

/*
 * Latent of FP8 cache rows (the reading of the low-precision cache the MLA
 * operator write-up names in its introduction and §5 tail: codes
 * dequantised on load).  Row r of `rows` (row_bytes each) holds d_c E4M3
 * codes, then d_R bf16 (the RoPE key, not read here), then d_c / blk fp32
 * scales; latent[r][i] = e4m3(code[i]) * scale[i / blk], in double.
 */
int mla_oracle_dequant_fp8(long n_rows, int d_c, int d_R, int blk, const uint8_t* rows, double* latent) {
  if (blk < 1 || d_c % blk != 0) return -1;
  const long row_bytes = d_c + 2L * d_R + 4L * (d_c / blk);
  for (long r = 0; r < n_rows; ++r) {
    const uint8_t* row = rows + r * row_bytes;
    for (int i = 0; i < d_c; ++i) {
      float sc;
      memcpy(&sc, row + d_c + 2 * d_R + 4 * (i / blk), sizeof sc);
      latent[r * d_c + i] = mla_oracle_e4m3(row[i]) * (double)sc;
    }
  }
  return 0;
}

/* Pointer to the cache row (d_c + d_R bf16) of token s of sequence b. */
static const uint16_t* cache_row(const uint16_t* cache, const int32_t* block_table,
                                 int max_pages, int P, int row_w, int b, int s) {
  int page = block_table[(size_t)b * max_pages + s / P];
  return cache + ((size_t)page * P + (size_t)(s % P)) * row_w;
}

int mla_oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Full decode, naive path, for the (b, h) pairs listed in sel[2*i], sel[2*i+1]
 * (i < n_sel), or for every (b, h) when sel == NULL.
 * Inputs (bf16 bits): q_nope [B,Lq,H,d_hc], q_rope [B,Lq,H,d_R],
 *   W_UK, W_UV [H,d_hc,d_g], cache [num_pages,P,d_c+d_R];
 *   block_table int32 [B,max_pages], seq_lens int32 [B].
 * Outputs (double, full shapes; only selected entries are written):
 *   out [B,Lq,H,d_hc], o_lat [B,Lq,H,d_g], lse [B,Lq,H] (any may be NULL).
 * Returns 0, or -1 on a bad argument (length, table entry out of range).
 */
int mla_oracle_decode(int B, int Lq, int H, int d_hc, int d_c, int d_R, int G,
                      int P, int max_pages, int num_pages, double scale, int causal,
                      const uint16_t* q_nope, const uint16_t* q_rope,
                      const uint16_t* W_UK, const uint16_t* W_UV,
                      const uint16_t* cache, const int32_t* block_table,
                      const int32_t* seq_lens, const int32_t* sel, int n_sel,
                      double* out, double* o_lat, double* lse, int nthreads) {
  const int d_g = d_c / G;
  const int row_w = d_c + d_R;
  if (G < 1 || d_c % G != 0 || H % G != 0) return -1;
  for (int b = 0; b < B; ++b) {
    int n = seq_lens[b];
    if (n < Lq || n < 1 || n > max_pages * P) return -1;
    for (int i = 0; i < (n + P - 1) / P; ++i) {
      int pg = block_table[(size_t)b * max_pages + i];
      if (pg < 0 || pg >= num_pages) return -1;
    }
  }
  const int total = sel ? n_sel : B * H;
  int err = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int it = 0; it < total; ++it) {
    const int b = sel ? sel[2 * it] : it / H;
    const int h = sel ? sel[2 * it + 1] : it % H;
    const int g = (h * G) / H;          /* contiguous head blocks per group */
    const int lat0 = g * d_g;
    const int n = seq_lens[b];
    double* score = (double*)malloc(sizeof(double) * (size_t)n);
    double* krow = (double*)malloc(sizeof(double) * (size_t)d_hc);
    double* qn = (double*)malloc(sizeof(double) * (size_t)d_hc);
    double* qr = (double*)malloc(sizeof(double) * (size_t)d_R);
    double* acc_out = (double*)malloc(sizeof(double) * (size_t)d_hc);
    double* acc_lat = (double*)malloc(sizeof(double) * (size_t)d_g);
    if (!score || !krow || !qn || !qr || !acc_out || !acc_lat) {
      err = 1;
    } else {
      const uint16_t* wk = W_UK + (size_t)h * d_hc * d_g;
      const uint16_t* wv = W_UV + (size_t)h * d_hc * d_g;
      for (int l = 0; l < Lq; ++l) {
        const size_t qi = ((size_t)b * Lq + l) * H + h;
        for (int d = 0; d < d_hc; ++d) qn[d] = bf16_to_double(q_nope[qi * d_hc + d]);
        for (int j = 0; j < d_R; ++j) qr[j] = bf16_to_double(q_rope[qi * d_R + j]);
        const int last = causal ? n - Lq + l : n - 1; /* last visible key */
        /* scores through the decompressed keys K_h[s] = W_UK[h] . c[s] */
        double mx = -INFINITY;
        for (int s = 0; s <= last; ++s) {
          const uint16_t* row = cache_row(cache, block_table, max_pages, P, row_w, b, s);
          for (int d = 0; d < d_hc; ++d) {
            double k = 0.0;
            for (int c = 0; c < d_g; ++c)
              k += bf16_to_double(wk[(size_t)d * d_g + c]) * bf16_to_double(row[lat0 + c]);
            krow[d] = k;
          }
          double sc = 0.0;
          for (int d = 0; d < d_hc; ++d) sc += qn[d] * krow[d];
          for (int j = 0; j < d_R; ++j) sc += qr[j] * bf16_to_double(row[d_c + j]);
          sc *= scale;
          score[s] = sc;
          if (sc > mx) mx = sc;
        }
        /* textbook softmax */
        double z = 0.0;
        for (int s = 0; s <= last; ++s) z += exp(score[s] - mx);
        for (int d = 0; d < d_hc; ++d) acc_out[d] = 0.0;
        for (int c = 0; c < d_g; ++c) acc_lat[c] = 0.0;
        /* out = sum_s p_s V_h[s], V_h[s] = W_UV[h] . c[s]; o_lat = sum_s p_s c[s] */
        for (int s = 0; s <= last; ++s) {
          const double p = exp(score[s] - mx) / z;
          const uint16_t* row = cache_row(cache, block_table, max_pages, P, row_w, b, s);
          for (int d = 0; d < d_hc; ++d) {
            double v = 0.0;
            for (int c = 0; c < d_g; ++c)
              v += bf16_to_double(wv[(size_t)d * d_g + c]) * bf16_to_double(row[lat0 + c]);
            acc_out[d] += p * v;
          }
          for (int c = 0; c < d_g; ++c) acc_lat[c] += p * bf16_to_double(row[lat0 + c]);
        }
        if (out)
          for (int d = 0; d < d_hc; ++d) out[qi * d_hc + d] = acc_out[d];
        if (o_lat)
          for (int c = 0; c < d_g; ++c) o_lat[qi * d_g + c] = acc_lat[c];
        if (lse) lse[qi] = mx + log(z);
      }
    }
    free(score); free(krow); free(qn); free(qr); free(acc_out); free(acc_lat);
  }
  return err ? -1 : 0;
}

/*
 * Scores of one query row (b, l, h) over all n = seq_lens[b] keys, by both
 * paths of the §4 equivalence script:
 *   s_naive[s]    = (q_nope . (W_UK[h] . c[s]) + q_rope . k_R[s]) * scale
 *   s_absorbed[s] = ((q_nope . W_UK[h]) . c[s] + q_rope . k_R[s]) * scale
 * Used only to check that matrix absorption leaves the scores unchanged.
 */
int mla_oracle_scores_both(int B, int Lq, int H, int d_hc, int d_c, int d_R, int G,
                           int P, int max_pages, double scale,
                           const uint16_t* q_nope, const uint16_t* q_rope,
                           const uint16_t* W_UK, const uint16_t* cache,
                           const int32_t* block_table, const int32_t* seq_lens,
                           int b, int l, int h, double* s_naive, double* s_absorbed) {
  const int d_g = d_c / G;
  const int row_w = d_c + d_R;
  const int g = (h * G) / H;
  const int lat0 = g * d_g;
  const int n = seq_lens[b];
  if (b < 0 || b >= B || l < 0 || l >= Lq || h < 0 || h >= H) return -1;
  const size_t qi = ((size_t)b * Lq + l) * H + h;
  const uint16_t* wk = W_UK + (size_t)h * d_hc * d_g;
  double* q_abs = (double*)malloc(sizeof(double) * (size_t)d_g);
  if (!q_abs) return -1;
  /* path B: absorb W_UK into the query once (einsum qhd,hdc->qhc) */
  for (int c = 0; c < d_g; ++c) {
    double a = 0.0;
    for (int d = 0; d < d_hc; ++d)
      a += bf16_to_double(q_nope[qi * d_hc + d]) * bf16_to_double(wk[(size_t)d * d_g + c]);
    q_abs[c] = a;
  }
  for (int s = 0; s < n; ++s) {
    const uint16_t* row = cache_row(cache, block_table, max_pages, P, row_w, b, s);
    double rope = 0.0;
    for (int j = 0; j < d_R; ++j)
      rope += bf16_to_double(q_rope[qi * d_R + j]) * bf16_to_double(row[d_c + j]);
    /* path A: decompress the key, then dot with the content query */
    double sa = 0.0;
    for (int d = 0; d < d_hc; ++d) {
      double k = 0.0;
      for (int c = 0; c < d_g; ++c)
        k += bf16_to_double(wk[(size_t)d * d_g + c]) * bf16_to_double(row[lat0 + c]);
      sa += bf16_to_double(q_nope[qi * d_hc + d]) * k;
    }
    double sb = 0.0;
    for (int c = 0; c < d_g; ++c) sb += q_abs[c] * bf16_to_double(row[lat0 + c]);
    s_naive[s] = (sa + rope) * scale;
    s_absorbed[s] = (sb + rope) * scale;
  }
  free(q_abs);
  return 0;
}

/*
 * Decode in the latent space from a given absorbed query: §4 "path B" (the
 * absorbed scores q_abs . c + q_R . k_R) carried through the softmax.  For
 * each selected (b, h) (all when sel == NULL) and each l:
 *   score_s = (q_cat[b,l,h,0:d_g] . c[s] + q_cat[b,l,h,d_g:] . k_R[s]) * scale
 * over the visible keys s <= n - Lq + l (all n keys if causal == 0), with
 * c[s] the latent slice of the head's group, then textbook softmax:
 *   o_lat = sum_s p_s c[s],   lse = max + log(sum_s exp(score_s - max)).
 * This is what the absorbed path holds before the W_UV projection.  It lets
 * the decode step be checked on a query given directly, e.g. one whose
 * scores are far larger than a unit-scale absorption produces.
 * q_cat bf16 bits [B,Lq,H,d_g+d_R]; outputs double o_lat [B,Lq,H,d_g] and
 * lse [B,Lq,H] (only selected entries written; either may be NULL).
 * Returns 0, or -1 on a bad argument (length, table entry out of range).
 */
int mla_oracle_decode_latent(int B, int Lq, int H, int d_c, int d_R, int G, int P,
                             int max_pages, int num_pages, double scale, int causal,
                             const uint16_t* q_cat, const uint16_t* cache,
                             const int32_t* block_table, const int32_t* seq_lens,
                             const int32_t* sel, int n_sel, double* o_lat, double* lse,
                             int nthreads) {
  const int d_g = d_c / G;
  const int row_w = d_c + d_R;
  const int d_q = d_g + d_R;
  if (G < 1 || d_c % G != 0 || H % G != 0) return -1;
  for (int b = 0; b < B; ++b) {
    int n = seq_lens[b];
    if (n < Lq || n < 1 || n > max_pages * P) return -1;
    for (int i = 0; i < (n + P - 1) / P; ++i) {
      int pg = block_table[(size_t)b * max_pages + i];
      if (pg < 0 || pg >= num_pages) return -1;
    }
  }
  const int total = sel ? n_sel : B * H;
  int err = 0;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int it = 0; it < total; ++it) {
    const int b = sel ? sel[2 * it] : it / H;
    const int h = sel ? sel[2 * it + 1] : it % H;
    const int lat0 = ((h * G) / H) * d_g;
    const int n = seq_lens[b];
    double* score = (double*)malloc(sizeof(double) * (size_t)n);
    double* q = (double*)malloc(sizeof(double) * (size_t)d_q);
    double* acc = (double*)malloc(sizeof(double) * (size_t)d_g);
    if (!score || !q || !acc) {
      err = 1;
    } else {
      for (int l = 0; l < Lq; ++l) {
        const size_t qi = ((size_t)b * Lq + l) * H + h;
        for (int j = 0; j < d_q; ++j) q[j] = bf16_to_double(q_cat[qi * d_q + j]);
        const int last = causal ? n - Lq + l : n - 1;
        double mx = -INFINITY;
        for (int s = 0; s <= last; ++s) {
          const uint16_t* row = cache_row(cache, block_table, max_pages, P, row_w, b, s);
          double sc = 0.0;
          for (int c = 0; c < d_g; ++c) sc += q[c] * bf16_to_double(row[lat0 + c]);
          for (int j = 0; j < d_R; ++j) sc += q[d_g + j] * bf16_to_double(row[d_c + j]);
          sc *= scale;
          score[s] = sc;
          if (sc > mx) mx = sc;
        }
        double z = 0.0;
        for (int s = 0; s <= last; ++s) z += exp(score[s] - mx);
        for (int c = 0; c < d_g; ++c) acc[c] = 0.0;
        for (int s = 0; s <= last; ++s) {
          const double p = exp(score[s] - mx) / z;
          const uint16_t* row = cache_row(cache, block_table, max_pages, P, row_w, b, s);
          for (int c = 0; c < d_g; ++c) acc[c] += p * bf16_to_double(row[lat0 + c]);
        }
        if (o_lat)
          for (int c = 0; c < d_g; ++c) o_lat[qi * d_g + c] = acc[c];
        if (lse) lse[qi] = mx + log(z);
      }
    }
    free(score); free(q); free(acc);
  }
  return err ? -1 : 0;
}

/*
 * Absorbed content query (§4 "path B"): q_abs[r,h,:] = q_nope[r,h,:] . W_UK[h]
 * for rows r = 0..R-1 (R = B*Lq).  Output double [R,H,d_g].
 */
int mla_oracle_absorb(int R, int H, int d_hc, int d_g, const uint16_t* q_nope,
                      const uint16_t* W_UK, double* q_abs) {
  for (int r = 0; r < R; ++r)
    for (int h = 0; h < H; ++h) {
      const uint16_t* q = q_nope + ((size_t)r * H + h) * d_hc;
      const uint16_t* w = W_UK + (size_t)h * d_hc * d_g;
      double* o = q_abs + ((size_t)r * H + h) * d_g;
      for (int c = 0; c < d_g; ++c) {
        double a = 0.0;
        for (int d = 0; d < d_hc; ++d)
          a += bf16_to_double(q[d]) * bf16_to_double(w[(size_t)d * d_g + c]);
        o[c] = a;
      }
    }
  return 0;
}

/*
 * Value up-projection applied after attention:
 *   out[r,h,d] = sum_c W_UV[h,d,c] * o_lat[r,h,c]
 * o_lat bf16 bits [R,H,d_g], W_UV bf16 bits [H,d_hc,d_g], out double [R,H,d_hc].
 */
int mla_oracle_project_uv(int R, int H, int d_hc, int d_g, const uint16_t* o_lat,
                          const uint16_t* W_UV, double* out) {
  for (int r = 0; r < R; ++r)
    for (int h = 0; h < H; ++h) {
      const uint16_t* x = o_lat + ((size_t)r * H + h) * d_g;
      const uint16_t* w = W_UV + (size_t)h * d_hc * d_g;
      double* o = out + ((size_t)r * H + h) * d_hc;
      for (int d = 0; d < d_hc; ++d) {
        double a = 0.0;
        for (int c = 0; c < d_g; ++c)
          a += bf16_to_double(w[(size_t)d * d_g + c]) * bf16_to_double(x[c]);
        o[d] = a;
      }
    }
  return 0;
}

/*
 * Log-sum-exp merge of S partial softmax results over disjoint key ranges
 * (the flash-decoding reduction): for each row r,
 *   L = log sum_k exp(lse[k,r]),  o[r,:] = sum_k exp(lse[k,r] - L) * o_part[k,r,:]
 * Partials with lse = -inf are empty ranges and contribute nothing; a row
 * whose partials are all empty gets L = -inf and o = 0.
 * o_part double [S,R,D], lse double [S,R] -> o double [R,D], L double [R].
 */
int mla_oracle_lse_merge(int S, int R, int D, const double* o_part, const double* lse,
                         double* o, double* L) {
  for (int r = 0; r < R; ++r) {
    double mx = -INFINITY;
    for (int k = 0; k < S; ++k)
      if (lse[(size_t)k * R + r] > mx) mx = lse[(size_t)k * R + r];
    for (int d = 0; d < D; ++d) o[(size_t)r * D + d] = 0.0;
    if (mx == -INFINITY) {
      L[r] = -INFINITY;
      continue;
    }
    double z = 0.0;
    for (int k = 0; k < S; ++k) z += exp(lse[(size_t)k * R + r] - mx);
    const double lr = mx + log(z);
    for (int k = 0; k < S; ++k) {
      const double w = exp(lse[(size_t)k * R + r] - lr);
      for (int d = 0; d < D; ++d) o[(size_t)r * D + d] += w * o_part[((size_t)k * R + r) * D + d];
    }
    L[r] = lr;
  }
  return 0;
}
