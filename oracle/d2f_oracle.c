/*
 * CPU oracle for the per-step hot path of Discrete Diffusion Forcing (D2F)
 * block-diffusion decoding.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing in the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header, table or helper with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "D2F: 확산 언어 모델이 KV 캐시를 얻고 자기회귀 모델보다 2.5배 빨라지는
 *        방법 (arXiv:2508.09192)" (llm-wiki.hwlabs.dev)
 *   [P2] "D2F 논문 리뷰: 확산 LLM이 자기회귀 모델보다 빠른 추론을 처음으로
 *        달성한 방식" (allinfo.ai.kr)
 *   [P3] "확산 언어 모델(Diffusion LLM)이란 무엇인가" (discuss.pytorch.kr)
 *
 * Every function below is the plain definition written out: no blocking, no
 * fusion, no reordering. Floating-point attention is done in double precision;
 * the commit widens logits to float (exact for bf16), accumulates the softmax
 * denominator in double and rounds the confidence to float.
 *
 * Parity pins for every function live in tests/ (brute force, closed forms,
 * hand-worked examples, invariants); none of them is "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_DT_BF16 0
#define ORACLE_DT_F32 1
#define ORACLE_DT_F64 2

/* Element access that widens the stored value exactly. bf16 is the upper half
 * of an IEEE binary32, so shifting its bits left by 16 gives the same number. */
static double load_elem(const void *base, int64_t idx, int dtype) {
  if (dtype == ORACLE_DT_BF16) {
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return (double)f;
  }
  if (dtype == ORACLE_DT_F64) return ((const double *)base)[idx];
  return (double)((const float *)base)[idx];
}

static float load_elem_f32(const void *base, int64_t idx, int dtype) {
  if (dtype == ORACLE_DT_BF16) {
    uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
    float f;
    memcpy(&f, &bits, sizeof f);
    return f;
  }
  return ((const float *)base)[idx];
}

/*
 * Block-causal attention of the active window over [cached context ; window].
 *
 * [P1] §블록 단위 인과 어텐션: the output is cut into fixed-size blocks; tokens
 * of one block attend to each other in both directions, a block attends only to
 * earlier blocks, so a finished block's K/V never change and go into an
 * ordinary KV cache. [P2] §쉽게 이해하기: a window of active blocks is decoded
 * together, each seeing its own block and the blocks before it.
 *
 * For sequence b with cached length C_b = ctx_len[b] and window rows
 * q_start[b] .. q_start[b+1]-1 (n_b rows, window block of row i is i / B), query
 * head h (KV head g = h / (Hq/Hkv)) of window row i sees:
 *   - every cached token t < C_b, stored in pool page page_table[b][t / B] at
 *     slot t % B, and
 *   - every window row i2 of the same sequence whose block i2 / B is not later
 *     than i / B.
 * Score = scale * <q, k>; output = softmax-weighted sum of v (max-subtracted
 * softmax in double); lse = natural-log normaliser (max + log(sum)).
 *
 * Operands are bf16, float or double (dtype 0 / 1 / 2), all of one type.
 * Layouts (row-major): q [total_q, Hq, D]; k_win, v_win [total_q, Hkv, D];
 * k_pool, v_pool [num_pages, Hkv, B, D]; page_table [batch, max_pages_per_seq];
 * out [total_q, Hq, D] double; lse [total_q, Hq] double (may be NULL).
 *
 * Returns 0, or a negative code: -1 bad sizes, -2 inconsistent q_start,
 * -3 page id out of range, -4 out of memory.
 */
static int block_attn_keys(const void *q, const void *k_win, const void *v_win,
                           const void *k_pool, const void *v_pool,
                           const int32_t *page_table, int max_pages_per_seq,
                           const int32_t *ctx_len, const int32_t *q_start,
                           int batch, int total_q, int num_heads_q,
                           int num_heads_kv, int head_dim, int block_size,
                           int num_pages, int dtype, double scale, double *out,
                           double *lse, int part, int nthreads) {
  if (batch < 0 || num_heads_q <= 0 || num_heads_kv <= 0 || head_dim <= 0 ||
      block_size <= 0 || num_heads_q % num_heads_kv != 0)
    return -1;
  if (q_start[0] != 0 || q_start[batch] != total_q) return -2;
  for (int b = 0; b < batch; ++b) {
    if (q_start[b + 1] < q_start[b]) return -2;
    if (ctx_len[b] < 0 || ctx_len[b] > max_pages_per_seq * block_size) return -1;
    int used_pages = (ctx_len[b] + block_size - 1) / block_size;
    for (int p = 0; p < used_pages; ++p) {
      int32_t pg = page_table[(int64_t)b * max_pages_per_seq + p];
      if (pg < 0 || pg >= num_pages) return -3;
    }
  }
  const int G = num_heads_q / num_heads_kv;
  const int H = num_heads_q, Hk = num_heads_kv, D = head_dim, B = block_size;
  const int64_t n_items = (int64_t)total_q * H;
  int err = 0;

#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads > 0 ? nthreads : 1)
  for (int64_t item = 0; item < n_items; ++item) {
    const int R = (int)(item / H); /* global window row */
    const int h = (int)(item % H);
    const int g = h / G;
    int b = 0;
    while (q_start[b + 1] <= R) ++b;
    const int i = R - q_start[b];
    const int n_b = q_start[b + 1] - q_start[b];
    const int C = ctx_len[b];
    const int max_keys = C + n_b;

    double *s = (double *)malloc(sizeof(double) * (size_t)(max_keys > 0 ? max_keys : 1));
    int64_t *koff = (int64_t *)malloc(sizeof(int64_t) * (size_t)(max_keys > 0 ? max_keys : 1));
    int *kwin = (int *)malloc(sizeof(int) * (size_t)(max_keys > 0 ? max_keys : 1));
    if (!s || !koff || !kwin) {
#pragma omp atomic write
      err = -4;
      free(s); free(koff); free(kwin);
      continue;
    }

    /* Build the visible key set K(i) (part 1: cached tokens only, 2: window only). */
    int nk = 0;
    for (int t = 0; part != 2 && t < C; ++t) {
      int32_t page = page_table[(int64_t)b * max_pages_per_seq + t / B];
      int slot = t % B;
      koff[nk] = (((int64_t)page * Hk + g) * B + slot) * D;
      kwin[nk] = 0;
      ++nk;
    }
    for (int i2 = 0; part != 1 && i2 < n_b; ++i2) {
      if (i2 / B <= i / B) {
        koff[nk] = ((int64_t)(q_start[b] + i2) * Hk + g) * D;
        kwin[nk] = 1;
        ++nk;
      }
    }

    const int64_t qoff = ((int64_t)R * H + h) * D;
    double mx = -INFINITY;
    for (int kk = 0; kk < nk; ++kk) {
      const void *kb = kwin[kk] ? k_win : k_pool;
      double dot = 0.0;
      for (int d = 0; d < D; ++d)
        dot += load_elem(q, qoff + d, dtype) * load_elem(kb, koff[kk] + d, dtype);
      s[kk] = scale * dot;
      if (s[kk] > mx) mx = s[kk];
    }
    double denom = 0.0;
    for (int kk = 0; kk < nk; ++kk) {
      s[kk] = exp(s[kk] - mx);
      denom += s[kk];
    }
    double *o = out + qoff;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (nk == 0) { /* no visible key (a cached part without cached tokens) */
      if (lse) lse[(int64_t)R * H + h] = -INFINITY;
      free(s);
      free(koff);
      free(kwin);
      continue;
    }
    for (int kk = 0; kk < nk; ++kk) {
      const void *vb = kwin[kk] ? v_win : v_pool;
      const double w = s[kk] / denom;
      for (int d = 0; d < D; ++d) o[d] += w * load_elem(vb, koff[kk] + d, dtype);
    }
    if (lse) lse[(int64_t)R * H + h] = mx + log(denom);
    free(s);
    free(koff);
    free(kwin);
  }
  return err;
}

int d2f_oracle_block_attn(const void *q, const void *k_win, const void *v_win,
                          const void *k_pool, const void *v_pool,
                          const int32_t *page_table, int max_pages_per_seq,
                          const int32_t *ctx_len, const int32_t *q_start,
                          int batch, int total_q, int num_heads_q,
                          int num_heads_kv, int head_dim, int block_size,
                          int num_pages, int dtype, double scale, double *out,
                          double *lse, int nthreads) {
  return block_attn_keys(q, k_win, v_win, k_pool, v_pool, page_table, max_pages_per_seq, ctx_len,
                         q_start, batch, total_q, num_heads_q, num_heads_kv, head_dim, block_size,
                         num_pages, dtype, scale, out, lse, 0, nthreads);
}

/*
 * The attention over one part of the keys, and the composition of a saved part
 * with the window part.
 *
 * [P3] §FlashBlock: 블록 외부 어텐션 캐싱: the attention output and normaliser over
 * the tokens outside the blocks being decoded are cached at one step; at the
 * next only the attention inside is recomputed, and the two are recombined in
 * log space as FlashAttention composes partial results.
 *
 * part 0: all visible keys (d2f_oracle_block_attn). part 1: the cached tokens
 * only (a row of a sequence with no cached token gets out 0, lse -inf). part 2:
 * the window keys only; with prev_out / prev_lse (a part-1 result, of this step
 * or an earlier one; double, same layouts as out / lse) the output is their
 * composition:
 *   out = (e^{lse_p} prev_out + e^{lse_w} out_w) / (e^{lse_p} + e^{lse_w}),
 *   lse = log(e^{lse_p} + e^{lse_w}),
 * computed with the larger of the two normalisers factored out. lse is
 * required for part 1 and part 2 (the composition needs it).
 */
int d2f_oracle_block_attn_part(const void *q, const void *k_win, const void *v_win,
                               const void *k_pool, const void *v_pool,
                               const int32_t *page_table, int max_pages_per_seq,
                               const int32_t *ctx_len, const int32_t *q_start,
                               int batch, int total_q, int num_heads_q,
                               int num_heads_kv, int head_dim, int block_size,
                               int num_pages, int dtype, double scale, int part,
                               const double *prev_out, const double *prev_lse,
                               double *out, double *lse, int nthreads) {
  if (part < 0 || part > 2 || (part != 0 && !lse)) return -1;
  const int rc = block_attn_keys(q, k_win, v_win, k_pool, v_pool, page_table, max_pages_per_seq,
                                 ctx_len, q_start, batch, total_q, num_heads_q, num_heads_kv,
                                 head_dim, block_size, num_pages, dtype, scale, out, lse, part,
                                 nthreads);
  if (rc != 0 || part != 2 || !prev_out || !prev_lse) return rc;
  const int64_t n_items = (int64_t)total_q * num_heads_q;
  const int D = head_dim;
  for (int64_t item = 0; item < n_items; ++item) {
    const double lp = prev_lse[item], lw = lse[item];
    const double M = lp > lw ? lp : lw;
    if (M == -INFINITY) continue;
    const double wp = lp == -INFINITY ? 0.0 : exp(lp - M);
    const double ww = lw == -INFINITY ? 0.0 : exp(lw - M);
    double *o = out + item * D;
    const double *po = prev_out + item * D;
    for (int d = 0; d < D; ++d) o[d] = (wp * po[d] + ww * o[d]) / (wp + ww);
    lse[item] = M + log(wp + ww);
  }
  return 0;
}

/*
 * Per-position confidence of a still-masked position.
 *
 * [P3] §양방향 어텐션과 사라진 KV 캐시 and §토큰 순서의 이론: LLaDA's default
 * low-confidence remasking ranks positions by the largest softmax probability
 * of the prediction. For a logit row l: m = max_v l_v, a = the lowest v with
 * l_v = m (greedy token), p_max = exp(m - logsumexp(l)) = 1 / sum_v exp(l_v - m).
 * Comparisons are exact in float; the sum is accumulated in double and the
 * reciprocal rounded to float once.
 */
static void row_confidence(const void *logits, int64_t row_off, int dtype,
                           int vocab, float *p_out, int32_t *a_out) {
  float m = -INFINITY;
  int32_t a = -1;
  for (int v = 0; v < vocab; ++v) {
    float x = load_elem_f32(logits, row_off + v, dtype);
    if (x > m || a < 0) {
      m = x;
      a = v;
    }
  }
  double S = 0.0;
  for (int v = 0; v < vocab; ++v) {
    double x = (double)load_elem_f32(logits, row_off + v, dtype);
    S += exp(x - (double)m);
  }
  *p_out = (float)(1.0 / S);
  *a_out = a;
}

/*
 * Alternative confidences of a still-masked position (same logit row).
 *
 * [P3] §토큰 순서의 이론: Dream ranks positions by negative entropy instead of the
 * largest probability, and the top-probability-margin ordering ranks them by the
 * difference between the largest and the second largest probability. [P3] §답을
 * 미리 안다: 조기 확정 디코딩(Prophet): the confidence gap is the difference
 * between the largest and the second largest logit.
 *
 * With m the largest logit, l2 the second largest (counted with multiplicity, so
 * l2 = m when the maximum occurs twice; -inf for a one-token vocabulary),
 * S = sum_v exp(l_v - m) and E = sum_v exp(l_v - m) (l_v - m):
 *   metric 1, negative entropy:  sum_v p_v log p_v = E / S - log S
 *   metric 2, probability margin: p_1 - p_2 = (1 - exp(l2 - m)) / S
 *   metric 3, logit gap:          m - l2
 * (p_v = exp(l_v - m) / S). Sums in double, each result rounded to float once;
 * the gap of two floats widened from bf16 is exact. A logit of -inf has
 * probability 0 and adds nothing to E. The greedy token is the lowest v with
 * l_v = m, as for metric 0.
 */
static void row_metric(const void *logits, int64_t row_off, int dtype, int vocab,
                       int metric, float *c_out, int32_t *a_out) {
  float m = -INFINITY, l2 = -INFINITY;
  int32_t a = -1;
  for (int v = 0; v < vocab; ++v) {
    const float x = load_elem_f32(logits, row_off + v, dtype);
    if (a < 0) {
      m = x;
      a = v;
    } else if (x > m) {
      l2 = m;
      m = x;
      a = v;
    } else if (x > l2) {
      l2 = x;
    }
  }
  double S = 0.0, E = 0.0;
  for (int v = 0; v < vocab; ++v) {
    const double x = (double)load_elem_f32(logits, row_off + v, dtype);
    if (x == -INFINITY) continue;
    const double t = exp(x - (double)m);
    S += t;
    E += t * (x - (double)m);
  }
  double c;
  if (metric == 1)
    c = E / S - log(S);
  else if (metric == 2)
    c = (1.0 - exp((double)l2 - (double)m)) / S;
  else
    c = (double)m - (double)l2;
  *c_out = (float)c;
  *a_out = a;
}

/*
 * Confidence commit with conservative / aggressive phases, then remasking.
 * `metric` picks the confidence: 0 the largest softmax probability (below), 1-3
 * the alternatives of row_metric (negative entropy, probability margin, logit
 * gap); tau is in the metric's own units.
 *
 * Early commit ([P3] §답을 미리 안다: 조기 확정 디코딩(Prophet): when the
 * confidence gap -- largest minus second largest logit -- over the answer region
 * exceeds a threshold, every remaining mask is filled with its argmax at once;
 * the threshold is lowered in stages (7.5, 5.0, 2.5) as decoding progresses).
 * With early_gap (per sequence, the caller's current threshold; NULL = off):
 * reading taken, the region is the sequence's window and its gap is the
 * smallest logit gap over the positions masked on entry; if that exceeds
 * early_gap[b] (strict), every masked position of b is committed with its
 * greedy token, its blocks' block_remaining become 0 and stopped[b] = 1; else
 * the block rules apply and stopped[b] = 0 (a sequence with nothing masked does
 * not stop). stopped may be NULL.
 *
 * [P2] §쉽게 이해하기 (pipelined decoding): a block that has just entered the
 * window is conservative and fixes only the tokens whose confidence is above
 * the threshold; once its predecessor has progressed enough it turns
 * aggressive and also fixes the relatively most confident token even when that
 * one is below the threshold; every token not fixed is masked again for the
 * next step. [P3] §양방향 어텐션과 사라진 KV 캐시: confidence is the maximum
 * softmax probability (low-confidence remasking).
 *
 * Readings where the pages are silent: "above" is strict (p > tau, in float);
 * the aggressive set is {p > tau} plus the masked position of highest p (lowest
 * position on ties); a block with no masked position commits nothing; positions
 * that were already committed are neither read nor changed.
 *
 * Window block jb covers rows jb*B .. jb*B+B-1 (q_start values are multiples of
 * B); its sequence b is the one whose rows contain it, tau[b] its threshold and
 * block_phase[jb] its phase (0 conservative, 1 aggressive).
 *
 * On return: committed rows get tokens[r] = a_r, masked[r] = 0; rows still
 * masked get tokens[r] = mask_id; rows not masked on entry keep their token.
 * conf_out[r] / argmax_out[r] = p_max / a for rows masked on entry and
 * -1 / -1 for the others (either may be NULL); block_remaining[jb] = masked
 * rows of block jb after the commit (may be NULL). logit_row (may be NULL)
 * maps position r to the logit row holding its prediction (identity when NULL).
 *
 * Returns 0, or -1 bad sizes, -2 inconsistent q_start, -3 logit row out of range.
 */
int d2f_oracle_commit_metric(const void *logits, int64_t row_stride, int dtype,
                             int vocab, int num_logit_rows, const int32_t *logit_row,
                             int32_t *tokens, uint8_t *masked, const int32_t *q_start,
                             const uint8_t *block_phase, const float *tau, int batch,
                             int total_q, int block_size, int32_t mask_id,
                             float *conf_out, int32_t *argmax_out,
                             int32_t *block_remaining, int metric, const float *early_gap,
                             uint8_t *stopped, int nthreads) {
  if (metric < 0 || metric > 3) return -1;
  if (batch < 0 || total_q < 0 || vocab <= 0 || block_size <= 0 ||
      block_size > 1024 || total_q % block_size != 0 || row_stride < vocab)
    return -1;
  if (q_start[0] != 0 || q_start[batch] != total_q) return -2;
  for (int b = 0; b < batch; ++b)
    if (q_start[b + 1] < q_start[b] || q_start[b] % block_size != 0) return -2;
  for (int r = 0; r < total_q; ++r) {
    int lr = logit_row ? logit_row[r] : r;
    if (masked[r] && (lr < 0 || lr >= num_logit_rows)) return -3;
  }

  float *conf = (float *)malloc(sizeof(float) * (size_t)(total_q > 0 ? total_q : 1));
  int32_t *amax = (int32_t *)malloc(sizeof(int32_t) * (size_t)(total_q > 0 ? total_q : 1));
  float *gap = (float *)malloc(sizeof(float) * (size_t)(total_q > 0 ? total_q : 1));
  if (!conf || !amax || !gap) {
    free(conf);
    free(amax);
    free(gap);
    return -4;
  }

  /* Confidence and greedy token of every position that is still masked. */
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
  for (int r = 0; r < total_q; ++r) {
    if (masked[r]) {
      int lr = logit_row ? logit_row[r] : r;
      if (metric == 0)
        row_confidence(logits, (int64_t)lr * row_stride, dtype, vocab, &conf[r], &amax[r]);
      else
        row_metric(logits, (int64_t)lr * row_stride, dtype, vocab, metric, &conf[r], &amax[r]);
      if (early_gap) {
        int32_t a2;
        row_metric(logits, (int64_t)lr * row_stride, dtype, vocab, 3, &gap[r], &a2);
      }
    } else {
      conf[r] = -1.0f;
      amax[r] = -1;
    }
  }

  /* Block-level commit decision, then remasking. */
  const int n_blocks = total_q / block_size;
  for (int jb = 0; jb < n_blocks; ++jb) {
    const int r0 = jb * block_size;
    int b = 0;
    while (q_start[b + 1] <= r0) ++b;
    const float t = tau[b];
    uint8_t commit[1024];
    int any_masked = 0;
    for (int u = 0; u < block_size; ++u) {
      const int r = r0 + u;
      commit[u] = 0;
      if (!masked[r]) continue;
      any_masked = 1;
      if (conf[r] > t) commit[u] = 1;
    }
    if (block_phase[jb] == 1 && any_masked) {
      int best = -1;
      for (int u = 0; u < block_size; ++u) {
        const int r = r0 + u;
        if (!masked[r]) continue;
        if (best < 0 || conf[r] > conf[r0 + best]) best = u;
      }
      commit[best] = 1;
    }
    int remaining = 0;
    for (int u = 0; u < block_size; ++u) {
      const int r = r0 + u;
      if (!masked[r]) continue;
      if (commit[u]) {
        tokens[r] = amax[r];
        masked[r] = 0;
      } else {
        tokens[r] = mask_id;
        ++remaining;
      }
    }
    if (block_remaining) block_remaining[jb] = remaining;
  }
  /* Early commit of a whole sequence (only with early_gap). */
  for (int b = 0; early_gap && b < batch; ++b) {
    float gmin = INFINITY;
    int any = 0;
    for (int r = q_start[b]; r < q_start[b + 1]; ++r)
      if (amax[r] >= 0) {  /* masked on entry */
        any = 1;
        if (gap[r] < gmin) gmin = gap[r];
      }
    const int stop = any && gmin > early_gap[b];
    if (stopped) stopped[b] = (uint8_t)stop;
    if (!stop) continue;
    for (int r = q_start[b]; r < q_start[b + 1]; ++r)
      if (masked[r]) {
        tokens[r] = amax[r];
        masked[r] = 0;
      }
    for (int jb = q_start[b] / block_size; jb < q_start[b + 1] / block_size; ++jb)
      if (block_remaining) block_remaining[jb] = 0;
  }
  if (!early_gap && stopped)
    for (int b = 0; b < batch; ++b) stopped[b] = 0;
  for (int r = 0; r < total_q; ++r) {
    if (conf_out) conf_out[r] = conf[r];
    if (argmax_out) argmax_out[r] = amax[r];
  }
  free(conf);
  free(amax);
  free(gap);
  return 0;
}

/* The commit with the largest softmax probability as confidence (metric 0). */
int d2f_oracle_commit(const void *logits, int64_t row_stride, int dtype,
                      int vocab, int num_logit_rows, const int32_t *logit_row,
                      int32_t *tokens, uint8_t *masked, const int32_t *q_start,
                      const uint8_t *block_phase, const float *tau, int batch,
                      int total_q, int block_size, int32_t mask_id,
                      float *conf_out, int32_t *argmax_out,
                      int32_t *block_remaining, int nthreads) {
  return d2f_oracle_commit_metric(logits, row_stride, dtype, vocab, num_logit_rows, logit_row,
                                  tokens, masked, q_start, block_phase, tau, batch, total_q,
                                  block_size, mask_id, conf_out, argmax_out, block_remaining,
                                  0, NULL, NULL, nthreads);
}

/*
 * Append finished blocks' K/V to the paged cache.
 *
 * [P1] §블록 단위 인과 어텐션 and §운영 관점 (KV 캐시 관리 방식): a completed
 * block's K/V are final and are stored permanently; with a paged cache whose
 * page is one block, completion of a block is the signal to persist it.
 *
 * For append a: rows src_row[a] .. src_row[a]+B-1 of k_win / v_win
 * ([total_q, Hkv, D]) are copied into page dst_page[a] of k_pool / v_pool
 * ([num_pages, Hkv, B, D]) as pool[dst][g][s][:] = win[src + s][g][:].
 * elem_bytes is 2 (bf16), 4 (float) or 8 (double); the copy is bitwise.
 * Returns 0, or -1 bad sizes, -3 page or row out of range.
 */
int d2f_oracle_kv_append(const void *k_win, const void *v_win,
                         const int32_t *src_row, const int32_t *dst_page,
                         int n_append, int total_q, void *k_pool, void *v_pool,
                         int num_heads_kv, int head_dim, int block_size,
                         int num_pages, int elem_bytes) {
  if (n_append < 0 || num_heads_kv <= 0 || head_dim <= 0 || block_size <= 0 ||
      (elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8))
    return -1;
  for (int a = 0; a < n_append; ++a) {
    if (dst_page[a] < 0 || dst_page[a] >= num_pages) return -3;
    if (src_row[a] < 0 || src_row[a] + block_size > total_q) return -3;
  }
  const int64_t row_bytes = (int64_t)head_dim * elem_bytes;
  for (int a = 0; a < n_append; ++a) {
    for (int g = 0; g < num_heads_kv; ++g) {
      for (int s = 0; s < block_size; ++s) {
        int64_t src = ((int64_t)(src_row[a] + s) * num_heads_kv + g) * row_bytes;
        int64_t dst = (((int64_t)dst_page[a] * num_heads_kv + g) * block_size + s) * row_bytes;
        memcpy((char *)k_pool + dst, (const char *)k_win + src, (size_t)row_bytes);
        memcpy((char *)v_pool + dst, (const char *)v_win + src, (size_t)row_bytes);
      }
    }
  }
  return 0;
}

/*
 * One step of the pipelined window scheduler, run after the commit of a step:
 * it turns the decode state left by that commit into the window of the next step.
 *
 * [P2] §쉽게 이해하기 (pipelined parallel decoding): an active window of blocks is
 * kept; when the progress of the window's last block passes a threshold a new
 * block is added behind it, so the window's size stays bounded; a new block
 * starts conservative (it commits only positions above the confidence threshold)
 * and turns aggressive (it also commits its most confident position) once the
 * block before it has progressed far enough; what is not committed stays masked.
 * [P1] §블록 단위 인과 어텐션 and §운영 관점: a completed block's K/V are final and
 * are persisted to the paged cache; block completion is the signal.
 *
 * Readings (the pages give neither values nor an order of these steps):
 *  - progress of a block = committed positions c out of B. "Passes the threshold"
 *    is c > tau_add * B and "far enough" is c >= tau_act * B, both products and
 *    comparisons in float. The block before the oldest window block is the cache
 *    (complete).
 *  - max_blocks bounds every block whose rows a step computes, including complete
 *    blocks waiting for their append. At most one block enters a sequence's
 *    window per step; an empty window takes one if any are left
 *    (next_block < gen_blocks) and the sequence was not stopped by the early
 *    commit.
 *  - a block that completed is appended during the next step (whose forward pass
 *    computes its K/V from final tokens), and only as part of a complete oldest
 *    prefix of the window (the cache stays in order). The blocks appended during
 *    a step leave the window at the next call (n_leaving), and ctx_len grows by B
 *    for each.
 *  - pages are taken from the top of the free list (free_pages[free_count - 1]
 *    first) in the order (sequence, block); the page of the i-th appended block of
 *    sequence b is written to page_table[b][ctx_len[b] / B + i] at once. A block
 *    that gets no page (list empty, or the page-table row full) stays in the
 *    window and err = 7.
 *
 * State, packed like the rest of the path (window rows of sequence b are
 * q_start[b] .. q_start[b+1]-1, block by block, oldest first), all in/out unless
 * said: q_start [batch+1]; tokens [capacity]; masked [capacity]; ctx_len [batch];
 * page_table [batch][max_pages_per_seq]; next_block [batch] (generation blocks
 * that have entered so far); gen_blocks [batch] (in); n_leaving [batch];
 * stopped [batch] (in, may be NULL); free_pages (in) and free_count.
 * Out: block_phase [capacity / B] (1 = aggressive); row_pos [capacity] (position
 * of the row's token in its sequence, -1 past the window); app_src / app_dst /
 * n_append (the append list of the next step: first window row of the block in
 * the new layout, its page). Rows past the new window: tokens = mask_id,
 * masked = 0, row_pos = -1; their blocks' phase 0.
 *
 * Returns 0; -1 bad sizes (nothing written); -2 inconsistent state (a window not
 * made of whole blocks, beyond capacity or longer than max_blocks, n_leaving
 * larger than the window, ctx_len negative or not a multiple of B): nothing
 * written. *err (first error wins, 0 = none) takes 7 when a block gets no page.
 */
int d2f_oracle_window_step(int batch, int block_size, int max_blocks, int capacity,
                           int max_pages_per_seq, int32_t mask_id, float tau_add, float tau_act,
                           int32_t *q_start, int32_t *tokens, uint8_t *masked,
                           uint8_t *block_phase, int32_t *row_pos, int32_t *ctx_len,
                           int32_t *page_table, int32_t *next_block, const int32_t *gen_blocks,
                           int32_t *n_leaving, const uint8_t *stopped,
                           const int32_t *free_pages, int32_t *free_count,
                           int32_t *app_src, int32_t *app_dst, int32_t *n_append, int32_t *err) {
  const int B = block_size;
  if (batch < 0 || B < 1 || max_blocks < 1 || capacity < 0 || capacity % B != 0 ||
      (long long)batch * max_blocks * B > capacity || max_pages_per_seq < 0 || *free_count < 0)
    return -1;
  /* the state must be consistent before anything is changed */
  if (q_start[0] != 0) return -2;
  for (int b = 0; b < batch; ++b) {
    const int n = q_start[b + 1] - q_start[b];
    if (n < 0 || n % B != 0 || n / B > max_blocks || q_start[b + 1] > capacity) return -2;
    if (n_leaving[b] < 0 || n_leaving[b] > n / B) return -2;
    if (ctx_len[b] < 0 || ctx_len[b] % B != 0) return -2;
  }
  /* the rows of the old window, read before any is overwritten */
  const int old_rows = q_start[batch];
  int32_t *tok0 = (int32_t *)malloc(sizeof(int32_t) * (size_t)(old_rows > 0 ? old_rows : 1));
  uint8_t *msk0 = (uint8_t *)malloc((size_t)(old_rows > 0 ? old_rows : 1));
  int32_t *qs0 = (int32_t *)malloc(sizeof(int32_t) * (size_t)(batch + 1));
  int *committed = (int *)malloc(sizeof(int) * (size_t)(max_blocks + 1));
  if (!tok0 || !msk0 || !qs0 || !committed) {
    free(tok0);
    free(msk0);
    free(qs0);
    free(committed);
    return -1;
  }
  memcpy(tok0, tokens, sizeof(int32_t) * (size_t)old_rows);
  memcpy(msk0, masked, (size_t)old_rows);
  memcpy(qs0, q_start, sizeof(int32_t) * (size_t)(batch + 1));

  int free_left = *free_count, n_app = 0, row = 0;
  for (int b = 0; b < batch; ++b) {
    const int old_blocks = (qs0[b + 1] - qs0[b]) / B;
    /* 1. the blocks appended during the step just run leave the window */
    const int nl = n_leaving[b];
    ctx_len[b] += nl * B;
    const int first_old = qs0[b] / B + nl; /* oldest surviving block (old layout) */
    const int n_surv = old_blocks - nl;
    /* committed positions of each block of the new window (a new block: none) */
    for (int k = 0; k < n_surv; ++k) {
      int c = 0;
      for (int u = 0; u < B; ++u) c += msk0[(first_old + k) * B + u] == 0;
      committed[k] = c;
    }
    /* 2. a new block behind the last one */
    const int is_stopped = stopped != NULL && stopped[b] != 0;
    int add = !is_stopped && next_block[b] < gen_blocks[b] && n_surv < max_blocks;
    if (add && n_surv > 0) add = (float)committed[n_surv - 1] > tau_add * (float)B;
    const int n_new = n_surv + add;
    if (add) committed[n_surv] = 0;
    q_start[b] = row;
    /* 3. the complete oldest blocks are appended during the next step */
    int want = 0;
    while (want < n_surv && committed[want] == B) ++want;
    int granted = 0;
    for (int i = 0; i < want; ++i) {
      const int slot = ctx_len[b] / B + i;
      if (free_left == 0 || slot >= max_pages_per_seq) {
        if (*err == 0) *err = 7;
        break;
      }
      const int page = free_pages[--free_left];
      page_table[(int64_t)b * max_pages_per_seq + slot] = page;
      app_src[n_app] = row + i * B;
      app_dst[n_app] = page;
      ++n_app;
      ++granted;
    }
    n_leaving[b] = granted;
    /* 4. phases and rows of the new window */
    for (int k = 0; k < n_new; ++k) {
      const int pred = k == 0 ? B : committed[k - 1];
      block_phase[row / B] = (float)pred >= tau_act * (float)B ? 1 : 0;
      for (int u = 0; u < B; ++u, ++row) {
        if (k < n_surv) {
          tokens[row] = tok0[(first_old + k) * B + u];
          masked[row] = msk0[(first_old + k) * B + u];
        } else {
          tokens[row] = mask_id;
          masked[row] = 1;
        }
        row_pos[row] = ctx_len[b] + k * B + u;
      }
    }
    next_block[b] += add;
  }
  q_start[batch] = row;
  for (int r = row; r < capacity; ++r) {
    tokens[r] = mask_id;
    masked[r] = 0;
    row_pos[r] = -1;
    if (r % B == 0) block_phase[r / B] = 0;
  }
  *free_count = free_left;
  *n_append = n_app;
  free(tok0);
  free(msk0);
  free(qs0);
  free(committed);
  return 0;
}
