/*
 * ringattn_oracle.c -- float64 CPU oracle for ring attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, plain reference that the
 * CUDA path is checked against.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table
 * or helper with the CUDA library, and it never includes anything from it.
 *
 * Sources (web pages on ring attention; cited by page title and section):
 *   [GRA]  "GPU Ring Attention" essay (aicassindra.com, gpu_ring_attention)
 *   [ZQ]   "Ring attention" explainer/quiz page (zenaique.com, attn-ring-attention)
 *   [RA-CN] "Ring Attention：把超长序列沿设备环流动" (charlestar.github.io)
 *
 * What it computes:
 *   - dense attention by its plain definition (the ring reaches exactly this
 *     result: [GRA] "Why partial results are allowed to merge"; [RA-CN]
 *     section "局部 Softmax 为什么不能直接相加", last paragraph);
 *   - a separate simulation of the P-step ring with per-row online-softmax
 *     states (m, l, O~) and the exact rescale merge ([RA-CN] "环是怎样工作的"
 *     and "局部 Softmax 为什么不能直接相加"; [GRA] "One lap around the ring");
 *   - the per-block partial state, the standalone merge of two states, and
 *     the (wrong) naive sum of per-block softmaxes used as a negative check.
 *
 * Readings where the pages are silent (their display formulas were lost):
 *   - scale = 1/sqrt(d); lse is the natural log of the sum of exp of the
 *     scaled scores; an empty row has state (m=-inf, l=0, O~=0) and a merge
 *     with an m=-inf side gives that side weight 0;
 *   - finalize: out = O~ / l, lse = m + ln(l);
 *   - layouts: contiguous pos(r,i) = r*n + i ([RA-CN] "位置编码必须使用全局位置");
 *     striped pos(r,i) = i*P + r (token t goes to shard t mod P);
 *     zigzag: the sequence cut into 2P chunks of c = n/2 tokens, shard r
 *     holding chunk r then chunk 2P-1-r ([GRA] "Striping the sequence to
 *     flatten the triangle"), local rows in that order;
 *   - causal: key position <= query position;
 *   - sliding window W > 0 (with the causal mask): a query also drops the
 *     keys W or more positions behind it, i.e. it sees itself and the W-1
 *     tokens before it ([RA-CN] "正确性测试应覆盖哪些边界" lists
 *     sliding-window masks among the cases to cover; the window is the
 *     usual causal local-attention window).
 *   - segments (sequence packing, [RA-CN] "正确性测试应覆盖哪些边界": several
 *     documents packed into one sequence must not attend to each other):
 *     seg[t] is the document of position t (NULL: one document); a pair is
 *     allowed only inside one document, on top of the causal rule and the
 *     window.  A valid-length mask (padding at the tail) is the case where
 *     the padding forms a document of its own.
 *
 * All inputs Q, K, V are bf16 bit patterns (uint16) in natural token order,
 * laid out [BH][N][d]; they are widened exactly to double.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_LAYOUT_CONTIGUOUS 0
#define ORACLE_LAYOUT_STRIPED 1
#define ORACLE_LAYOUT_ZIGZAG 2

static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

/* Number of threads an OpenMP parallel region would use now. */
int oracle_max_threads(int nthreads) {
  set_threads(nthreads);
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Global token position of local row i of shard r ([RA-CN] "位置编码必须使用全局位置"
 * for the contiguous map; the striped map sends token t to shard t mod P). */
long oracle_position(int layout, long n, int P, int r, long i) {
  if (layout == ORACLE_LAYOUT_STRIPED) return i * (long)P + r;
  if (layout == ORACLE_LAYOUT_ZIGZAG) {
    const long c = n / 2;
    return i < c ? (long)r * c + i : (long)(2 * P - 1 - r) * c + (i - c);
  }
  return (long)r * n + i;
}

/* The inverse: the shard holding global position t and its local row. */
void oracle_owner(int layout, long n, int P, long t, int* r, long* i) {
  if (layout == ORACLE_LAYOUT_STRIPED) {
    *r = (int)(t % P);
    *i = t / P;
  } else if (layout == ORACLE_LAYOUT_ZIGZAG) {
    const long c = n / 2, chunk = t / c;
    *r = chunk < P ? (int)chunk : (int)(2 * P - 1 - chunk);
    *i = t % c + (chunk < P ? 0 : c);
  } else {
    *r = (int)(t / n);
    *i = t % n;
  }
}

/* Shapes a layout accepts: N divisible by P, and for zigzag by 2P. */
static int layout_ok(int layout, long N, int P) {
  if (P <= 0 || N % P != 0) return 0;
  if (layout == ORACLE_LAYOUT_ZIGZAG) return (N / P) % 2 == 0;
  return layout == ORACLE_LAYOUT_CONTIGUOUS || layout == ORACLE_LAYOUT_STRIPED;
}

/* The K/V block that rank r holds at ring step s: rank r sends to r+1 and
 * receives from r-1, starting from its own block ([GRA] "One lap around the
 * ring"; [RA-CN] "环是怎样工作的", the 4-device walk-through). */
int oracle_block_at(int P, int r, int s) {
  int j = (r - s) % P;
  if (j < 0) j += P;
  return j;
}

static int allowed(int causal, long window, const long* seg, long pos_q, long pos_k) {
  if (seg && seg[pos_q] != seg[pos_k]) return 0;
  if (window > 0 && pos_q - pos_k >= window) return 0;
  return !causal || pos_k <= pos_q;
}

static double dot_q_k(const uint16_t* q, const uint16_t* k, int d) {
  double acc = 0.0;
  for (int c = 0; c < d; ++c) acc += widen_bf16(q[c]) * widen_bf16(k[c]);
  return acc;
}

/*
 * Dense attention, plain definition, for a list of query positions.
 *   s_k   = (q . k) / sqrt(d)          for every allowed key k
 *   lse   = log sum_k exp(s_k)         (computed with the row max subtracted)
 *   out   = sum_k exp(s_k - lse) v_k
 * rows == NULL means every position 0..N-1 (nrows must equal N then).
 * out is [BH][nrows][d], lse is [BH][nrows].
 */
int oracle_dense_rows(int BH, long N, int d, int causal, long window, const long* seg, const uint16_t* q,
                      const uint16_t* k, const uint16_t* v, long nrows,
                      const long* rows, double* out, double* lse,
                      int nthreads) {
  if (BH <= 0 || N <= 0 || d <= 0 || nrows < 0) return -1;
  set_threads(nthreads);
  const double scale = 1.0 / sqrt((double)d);
  long total = (long)BH * nrows;
  int failed = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    if (!s) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 4)
    for (long idx = 0; idx < total; ++idx) {
      if (!s) continue;
      long bh = idx / nrows, ri = idx % nrows;
      long t = rows ? rows[ri] : ri;
      const uint16_t* qrow = q + ((size_t)bh * N + t) * d;
      const uint16_t* kb = k + (size_t)bh * N * d;
      const uint16_t* vb = v + (size_t)bh * N * d;
      double m = -INFINITY;
      for (long kk = 0; kk < N; ++kk) {
        if (!allowed(causal, window, seg, t, kk)) continue;
        s[kk] = scale * dot_q_k(qrow, kb + (size_t)kk * d, d);
        if (s[kk] > m) m = s[kk];
      }
      double sum = 0.0;
      for (long kk = 0; kk < N; ++kk)
        if (allowed(causal, window, seg, t, kk)) sum += exp(s[kk] - m);
      double l = m + log(sum);
      double* o = out + (size_t)idx * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (long kk = 0; kk < N; ++kk) {
        if (!allowed(causal, window, seg, t, kk)) continue;
        double w = exp(s[kk] - l);
        const uint16_t* vr = vb + (size_t)kk * d;
        for (int c = 0; c < d; ++c) o[c] += w * widen_bf16(vr[c]);
      }
      lse[idx] = l;
    }
    free(s);
  }
  return failed ? -2 : 0;
}

/*
 * Partial state of one query row against one K/V block, by definition
 * ([RA-CN] "局部 Softmax 为什么不能直接相加": per row the running max m, the exp
 * sum l scaled by that max, and the unnormalised value sum O~):
 *   m  = max over allowed keys of s_k        (-inf if none allowed)
 *   l  = sum exp(s_k - m)
 *   O~ = sum exp(s_k - m) v_k
 * kpos[k] is the global position of key k of the block.
 */
static void row_block_state(const uint16_t* qrow, long pos_q, const uint16_t* kb,
                            const uint16_t* vb, const long* kpos, long nk, int d,
                            int causal, long window, const long* seg, double scale, double* s, double* m_out,
                            double* l_out, double* o_out, long* visit_row) {
  double m = -INFINITY;
  for (long kk = 0; kk < nk; ++kk) {
    if (!allowed(causal, window, seg, pos_q, kpos[kk])) continue;
    s[kk] = scale * dot_q_k(qrow, kb + (size_t)kk * d, d);
    if (s[kk] > m) m = s[kk];
  }
  double l = 0.0;
  for (int c = 0; c < d; ++c) o_out[c] = 0.0;
  if (m != -INFINITY) {
    for (long kk = 0; kk < nk; ++kk) {
      if (!allowed(causal, window, seg, pos_q, kpos[kk])) continue;
      double w = exp(s[kk] - m);
      l += w;
      const uint16_t* vr = vb + (size_t)kk * d;
      for (int c = 0; c < d; ++c) o_out[c] += w * widen_bf16(vr[c]);
      if (visit_row) visit_row[kpos[kk]] += 1;
    }
  }
  *m_out = m;
  *l_out = l;
}

/*
 * Merge of two online-softmax states into (m, l, O~) ([GRA] "Why partial
 * results are allowed to merge": both accumulators are rescaled by the exp of
 * the difference between the old and the new maximum, then added; [ZQ]: the
 * running output is rescaled by exp(old_max - new_max)).
 *   m = max(ma, mb); a = exp(ma - m); b = exp(mb - m)  (0 for an -inf side)
 *   l = a la + b lb;  O~ = a O~a + b O~b
 */
static void merge_pair(double ma, double la, const double* oa, double mb,
                       double lb, const double* ob, int d, double* m,
                       double* l, double* o) {
  double mm = ma > mb ? ma : mb;
  double a = (ma == -INFINITY) ? 0.0 : exp(ma - mm);
  double b = (mb == -INFINITY) ? 0.0 : exp(mb - mm);
  *m = mm;
  *l = a * la + b * lb;
  for (int c = 0; c < d; ++c) o[c] = a * oa[c] + b * ob[c];
}

/*
 * Ring simulation ([RA-CN] "环是怎样工作的": the forward as a loop over
 * world_size steps that computes a block partial and merges it into the local
 * state, then finalizes; [GRA] "One lap around the ring").
 * P virtual ranks; rank r owns the query rows of shard r.  At step s it holds
 * block j = (r - s) mod P, computes the block partial of its rows against it
 * and merges that into its running state; after P steps it finalizes
 *   out = O~ / l,   lse = m + ln l.
 * rows: global query positions to simulate (NULL = all N).  out/lse are
 * indexed like oracle_dense_rows.  visits (NULL or [BH][N][N] counters)
 * receives +1 for every (query, key) pair the simulation used.
 */
int oracle_ring_rows(int BH, long N, int d, int P, int causal, long window, const long* seg, int layout,
                     const uint16_t* q, const uint16_t* k, const uint16_t* v,
                     long nrows, const long* rows, double* out, double* lse,
                     long* visits, int nthreads) {
  if (BH <= 0 || N <= 0 || d <= 0 || !layout_ok(layout, N, P) || nrows < 0)
    return -1;
  set_threads(nthreads);
  const long n = N / P;
  const double scale = 1.0 / sqrt((double)d);
  long total = (long)BH * nrows;
  int failed = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    long* kpos = (long*)malloc(sizeof(long) * (size_t)n);
    uint16_t* kblk = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * d);
    uint16_t* vblk = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * d);
    double* ob = (double*)malloc(sizeof(double) * (size_t)d);
    double* ost = (double*)malloc(sizeof(double) * (size_t)d);
    double* otmp = (double*)malloc(sizeof(double) * (size_t)d);
    int ok = s && kpos && kblk && vblk && ob && ost && otmp;
    if (!ok) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (long idx = 0; idx < total; ++idx) {
      if (!ok) continue;
      long bh = idx / nrows, ri = idx % nrows;
      long t = rows ? rows[ri] : ri;
      /* which rank owns query position t, and its local row */
      int r;
      long i;
      oracle_owner(layout, n, P, t, &r, &i);
      const uint16_t* qrow =
          q + ((size_t)bh * N + oracle_position(layout, n, P, r, i)) * d;
      long* visit_row = visits ? visits + ((size_t)bh * N + t) * N : NULL;
      double m = -INFINITY, l = 0.0;
      for (int c = 0; c < d; ++c) ost[c] = 0.0;
      for (int step = 0; step < P; ++step) {
        int j = oracle_block_at(P, r, step);
        /* the block as it would travel: rows of shard j, in local order */
        for (long kk = 0; kk < n; ++kk) {
          long pk = oracle_position(layout, n, P, j, kk);
          kpos[kk] = pk;
          memcpy(kblk + (size_t)kk * d, k + ((size_t)bh * N + pk) * d,
                 sizeof(uint16_t) * d);
          memcpy(vblk + (size_t)kk * d, v + ((size_t)bh * N + pk) * d,
                 sizeof(uint16_t) * d);
        }
        double mb, lb;
        row_block_state(qrow, t, kblk, vblk, kpos, n, d, causal, window, seg, scale, s, &mb,
                        &lb, ob, visit_row);
        double mn, ln;
        merge_pair(m, l, ost, mb, lb, ob, d, &mn, &ln, otmp);
        m = mn;
        l = ln;
        memcpy(ost, otmp, sizeof(double) * d);
      }
      double* o = out + (size_t)idx * d;
      for (int c = 0; c < d; ++c) o[c] = ost[c] / l;
      lse[idx] = m + log(l);
    }
    free(s);
    free(kpos);
    free(kblk);
    free(vblk);
    free(ob);
    free(ost);
    free(otmp);
  }
  return failed ? -2 : 0;
}

/*
 * Block partial state of shard r's query rows against K/V block j, with the
 * global-position mask ([RA-CN] "Causal Attention 让环不再完全对称": skip a
 * strictly-future block, mask a block on the diagonal, else no mask).
 * q_shard, k_block, v_block are shard-major [BH][n][d] bf16 bit patterns.
 * Outputs m, l [BH][n] and o [BH][n][d] as defined in row_block_state.
 */
int oracle_block_partial(int BH, long n, int d, int P, int causal, long window, const long* seg, int layout,
                         int r, int j, const uint16_t* q_shard,
                         const uint16_t* k_block, const uint16_t* v_block,
                         double* m, double* l, double* o, int nthreads) {
  if (BH <= 0 || n <= 0 || d <= 0 || !layout_ok(layout, n * (long)P, P) ||
      r < 0 || r >= P || j < 0 || j >= P)
    return -1;
  set_threads(nthreads);
  const double scale = 1.0 / sqrt((double)d);
  long total = (long)BH * n;
  int failed = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    long* kpos = (long*)malloc(sizeof(long) * (size_t)n);
    int ok = s && kpos;
    if (!ok) {
#pragma omp atomic write
      failed = 1;
    }
    if (ok)
      for (long kk = 0; kk < n; ++kk)
        kpos[kk] = oracle_position(layout, n, P, j, kk);
#pragma omp for schedule(dynamic, 4)
    for (long idx = 0; idx < total; ++idx) {
      if (!ok) continue;
      long bh = idx / n, i = idx % n;
      row_block_state(q_shard + (size_t)idx * d,
                      oracle_position(layout, n, P, r, i),
                      k_block + (size_t)bh * n * d, v_block + (size_t)bh * n * d,
                      kpos, n, d, causal, window, seg, scale, s, &m[idx], &l[idx],
                      o + (size_t)idx * d, NULL);
    }
    free(s);
    free(kpos);
  }
  return failed ? -2 : 0;
}

/*
 * Standalone merge of two fp32 states (as a GPU produces them), in float64.
 * Inputs: rows x {m, l} and rows x d for O~, per side.  Outputs in double.
 */
int oracle_merge_states(long rows, int d, const float* ma, const float* la,
                        const float* oa, const float* mb, const float* lb,
                        const float* ob, double* m, double* l, double* o) {
  if (rows < 0 || d <= 0) return -1;
  double* ta = (double*)malloc(sizeof(double) * (size_t)d);
  double* tb = (double*)malloc(sizeof(double) * (size_t)d);
  if (!ta || !tb) {
    free(ta);
    free(tb);
    return -2;
  }
  for (long x = 0; x < rows; ++x) {
    for (int c = 0; c < d; ++c) {
      ta[c] = (double)oa[(size_t)x * d + c];
      tb[c] = (double)ob[(size_t)x * d + c];
    }
    merge_pair((double)ma[x], (double)la[x], ta, (double)mb[x], (double)lb[x],
               tb, d, &m[x], &l[x], o + (size_t)x * d);
  }
  free(ta);
  free(tb);
  return 0;
}

/* Same merge on double states: a <- merge(a, b), in place.  Used to check that
 * the merge is order independent (associative and commutative). */
int oracle_merge_inplace(long rows, int d, double* ma, double* la, double* oa,
                         const double* mb, const double* lb, const double* ob) {
  if (rows < 0 || d <= 0) return -1;
  double* t = (double*)malloc(sizeof(double) * (size_t)d);
  if (!t) return -2;
  for (long x = 0; x < rows; ++x) {
    double m, l;
    merge_pair(ma[x], la[x], oa + (size_t)x * d, mb[x], lb[x],
               ob + (size_t)x * d, d, &m, &l, t);
    ma[x] = m;
    la[x] = l;
    memcpy(oa + (size_t)x * d, t, sizeof(double) * d);
  }
  free(t);
  return 0;
}

/* Finalize states: out = O~/l, lse = m + ln l (an empty row gives out = 0 and
 * lse = -inf). */
int oracle_finalize(long rows, int d, const double* m, const double* l,
                    const double* o, double* out, double* lse) {
  if (rows < 0 || d <= 0) return -1;
  for (long x = 0; x < rows; ++x) {
    if (l[x] == 0.0) {
      for (int c = 0; c < d; ++c) out[(size_t)x * d + c] = 0.0;
      lse[x] = -INFINITY;
      continue;
    }
    for (int c = 0; c < d; ++c)
      out[(size_t)x * d + c] = o[(size_t)x * d + c] / l[x];
    lse[x] = m[x] + log(l[x]);
  }
  return 0;
}

/*
 * The wrong combination the pages warn against ([GRA] "Why partial results
 * are allowed to merge": naively summing partial outputs is wrong; [RA-CN]
 * "局部 Softmax 为什么不能直接相加": a softmax per block, outputs added):
 *   out_naive = sum over blocks j with an allowed key of softmax(S^(j)) V_j.
 * Natural order in and out, out is [BH][N][d].
 */
int oracle_naive_block_sum(int BH, long N, int d, int P, int causal, long window, const long* seg, int layout,
                           const uint16_t* q, const uint16_t* k,
                           const uint16_t* v, double* out) {
  if (BH <= 0 || N <= 0 || d <= 0 || !layout_ok(layout, N, P)) return -1;
  const long n = N / P;
  const double scale = 1.0 / sqrt((double)d);
  double* s = (double*)malloc(sizeof(double) * (size_t)n);
  long* kpos = (long*)malloc(sizeof(long) * (size_t)n);
  uint16_t* kblk = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * d);
  uint16_t* vblk = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)n * d);
  double* ob = (double*)malloc(sizeof(double) * (size_t)d);
  if (!s || !kpos || !kblk || !vblk || !ob) {
    free(s); free(kpos); free(kblk); free(vblk); free(ob);
    return -2;
  }
  for (int bh = 0; bh < BH; ++bh) {
    for (long t = 0; t < N; ++t) {
      double* o = out + ((size_t)bh * N + t) * d;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      const uint16_t* qrow = q + ((size_t)bh * N + t) * d;
      for (int j = 0; j < P; ++j) {
        for (long kk = 0; kk < n; ++kk) {
          long pk = oracle_position(layout, n, P, j, kk);
          kpos[kk] = pk;
          memcpy(kblk + (size_t)kk * d, k + ((size_t)bh * N + pk) * d,
                 sizeof(uint16_t) * d);
          memcpy(vblk + (size_t)kk * d, v + ((size_t)bh * N + pk) * d,
                 sizeof(uint16_t) * d);
        }
        double mb, lb;
        row_block_state(qrow, t, kblk, vblk, kpos, n, d, causal, window, seg, scale, s, &mb,
                        &lb, ob, NULL);
        if (lb > 0.0)
          for (int c = 0; c < d; ++c) o[c] += ob[c] / lb;
      }
    }
  }
  free(s); free(kpos); free(kblk); free(vblk); free(ob);
  return 0;
}

/* ------------------------------------------------------------------ backward
 *
 * The gradients of attention for an upstream gradient dO ([RA-CN] "Backward
 * 需要让梯度也沿环传播": every Q-K/V block interaction contributes a gradient;
 * the softmax statistics are restored from the saved per-row logsumexp and
 * the probabilities recomputed block by block, as in FlashAttention's
 * backward).  With P_tk = exp(s_tk - lse_t) over the allowed keys of query t:
 *   dV_k = sum_t P_tk dO_t
 *   dP_tk = dO_t . v_k
 *   D_t  = sum_k P_tk dP_tk = dO_t . O_t
 *   dS_tk = P_tk (dP_tk - D_t)
 *   dQ_t = scale sum_k dS_tk k_k
 *   dK_k = scale sum_t dS_tk q_t
 * (the chain rule through O = softmax(scale Q K^T) V; the derivative of a
 * softmax row p is diag(p) - p p^T, which gives the D_t term).
 */

/*
 * Dense backward by the definition above, from scratch (the forward's O and
 * lse are recomputed here in float64).  q, k, v, dout are bf16 bit patterns
 * [BH][N][d] in natural order; dq, dk, dv are [BH][N][d] doubles.
 * Two passes so that every output row has a single writer:
 *   pass 1, per query t: lse_t, O_t, D_t and dQ_t;
 *   pass 2, per key k:   dK_k and dV_k over the queries that see k.
 */
int oracle_dense_bwd(int BH, long N, int d, int causal, long window, const long* seg, const uint16_t* q,
                     const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                     double* dq, double* dk, double* dv, int nthreads) {
  if (BH <= 0 || N <= 0 || d <= 0) return -1;
  set_threads(nthreads);
  const double scale = 1.0 / sqrt((double)d);
  double* lse = (double*)malloc(sizeof(double) * (size_t)BH * N);
  double* D = (double*)malloc(sizeof(double) * (size_t)BH * N);
  if (!lse || !D) {
    free(lse);
    free(D);
    return -2;
  }
  int failed = 0;
  const long total = (long)BH * N;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    double* o = (double*)malloc(sizeof(double) * (size_t)d);
    const int ok = s && o;
    if (!ok) {
#pragma omp atomic write
      failed = 1;
    }
    /* pass 1: per query row */
#pragma omp for schedule(dynamic, 4)
    for (long idx = 0; idx < total; ++idx) {
      if (!ok) continue;
      const long bh = idx / N, t = idx % N;
      const uint16_t* qrow = q + (size_t)idx * d;
      const uint16_t* dorow = dout + (size_t)idx * d;
      const uint16_t* kb = k + (size_t)bh * N * d;
      const uint16_t* vb = v + (size_t)bh * N * d;
      double m = -INFINITY;
      for (long kk = 0; kk < N; ++kk) {
        if (!allowed(causal, window, seg, t, kk)) continue;
        s[kk] = scale * dot_q_k(qrow, kb + (size_t)kk * d, d);
        if (s[kk] > m) m = s[kk];
      }
      double sum = 0.0;
      for (long kk = 0; kk < N; ++kk)
        if (allowed(causal, window, seg, t, kk)) sum += exp(s[kk] - m);
      const double l = m + log(sum);
      lse[idx] = l;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (long kk = 0; kk < N; ++kk) {
        if (!allowed(causal, window, seg, t, kk)) continue;
        const double p = exp(s[kk] - l);
        for (int c = 0; c < d; ++c) o[c] += p * widen_bf16(vb[(size_t)kk * d + c]);
      }
      double Dt = 0.0;
      for (int c = 0; c < d; ++c) Dt += widen_bf16(dorow[c]) * o[c];
      D[idx] = Dt;
      double* g = dq + (size_t)idx * d;
      for (int c = 0; c < d; ++c) g[c] = 0.0;
      for (long kk = 0; kk < N; ++kk) {
        if (!allowed(causal, window, seg, t, kk)) continue;
        const double p = exp(s[kk] - l);
        const double ds = p * (dot_q_k(dorow, vb + (size_t)kk * d, d) - Dt);
        for (int c = 0; c < d; ++c) g[c] += scale * ds * widen_bf16(kb[(size_t)kk * d + c]);
      }
    }
    /* pass 2: per key row (the implicit barrier above makes lse and D ready) */
#pragma omp for schedule(dynamic, 4)
    for (long idx = 0; idx < total; ++idx) {
      if (!ok) continue;
      const long bh = idx / N, kk = idx % N;
      const uint16_t* krow = k + (size_t)idx * d;
      const uint16_t* vrow = v + (size_t)idx * d;
      double* gk = dk + (size_t)idx * d;
      double* gv = dv + (size_t)idx * d;
      for (int c = 0; c < d; ++c) gk[c] = gv[c] = 0.0;
      for (long t = 0; t < N; ++t) {
        if (!allowed(causal, window, seg, t, kk)) continue;
        const size_t row = (size_t)bh * N + t;
        const uint16_t* qrow = q + row * d;
        const uint16_t* dorow = dout + row * d;
        const double p = exp(scale * dot_q_k(qrow, krow, d) - lse[row]);
        const double ds = p * (dot_q_k(dorow, vrow, d) - D[row]);
        for (int c = 0; c < d; ++c) {
          gk[c] += scale * ds * widen_bf16(qrow[c]);
          gv[c] += p * widen_bf16(dorow[c]);
        }
      }
    }
    free(s);
    free(o);
  }
  free(lse);
  free(D);
  return failed ? -2 : 0;
}

/* lse_t and D_t = dO_t . O_t of one query row, by definition. */
static void row_lse_and_D(const uint16_t* qrow, const uint16_t* dorow, long t, const uint16_t* kb,
                          const uint16_t* vb, long N, int d, int causal, long window, const long* seg, double scale,
                          double* s, double* o, double* lse_out, double* D_out) {
  double m = -INFINITY;
  for (long kk = 0; kk < N; ++kk) {
    if (!allowed(causal, window, seg, t, kk)) continue;
    s[kk] = scale * dot_q_k(qrow, kb + (size_t)kk * d, d);
    if (s[kk] > m) m = s[kk];
  }
  double sum = 0.0;
  for (long kk = 0; kk < N; ++kk)
    if (allowed(causal, window, seg, t, kk)) sum += exp(s[kk] - m);
  const double l = m + log(sum);
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  for (long kk = 0; kk < N; ++kk) {
    if (!allowed(causal, window, seg, t, kk)) continue;
    const double p = exp(s[kk] - l);
    for (int c = 0; c < d; ++c) o[c] += p * widen_bf16(vb[(size_t)kk * d + c]);
  }
  double Dt = 0.0;
  for (int c = 0; c < d; ++c) Dt += widen_bf16(dorow[c]) * o[c];
  *lse_out = l;
  *D_out = Dt;
}

/*
 * The dense backward for sampled rows only: dQ at the query positions qrows
 * (dq is [BH][nq][d]) and dK, dV at the key positions krows (dk, dv are
 * [BH][nk][d]).  Same definition as oracle_dense_bwd; the statistics of each
 * query that a sampled key meets are recomputed on demand, so a key late in
 * a causal sequence (or any key under a sliding window) is cheap.
 */
int oracle_dense_bwd_rows(int BH, long N, int d, int causal, long window, const long* seg, const uint16_t* q,
                          const uint16_t* k, const uint16_t* v, const uint16_t* dout, long nq,
                          const long* qrows, long nk, const long* krows, double* dq, double* dk,
                          double* dv, int nthreads) {
  if (BH <= 0 || N <= 0 || d <= 0 || nq < 0 || nk < 0) return -1;
  set_threads(nthreads);
  const double scale = 1.0 / sqrt((double)d);
  int failed = 0;
  const long total = (long)BH * (nq + nk);
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    double* o = (double*)malloc(sizeof(double) * (size_t)d);
    const int ok = s && o;
    if (!ok) {
#pragma omp atomic write
      failed = 1;
    }
#pragma omp for schedule(dynamic, 1)
    for (long idx = 0; idx < total; ++idx) {
      if (!ok) continue;
      const long bh = idx / (nq + nk), x = idx % (nq + nk);
      const uint16_t* qb = q + (size_t)bh * N * d;
      const uint16_t* kb = k + (size_t)bh * N * d;
      const uint16_t* vb = v + (size_t)bh * N * d;
      const uint16_t* ob = dout + (size_t)bh * N * d;
      if (x < nq) {
        const long t = qrows[x];
        double l, Dt;
        row_lse_and_D(qb + (size_t)t * d, ob + (size_t)t * d, t, kb, vb, N, d, causal, window, seg, scale, s, o,
                      &l, &Dt);
        double* g = dq + ((size_t)bh * nq + x) * d;
        for (int c = 0; c < d; ++c) g[c] = 0.0;
        for (long kk = 0; kk < N; ++kk) {
          if (!allowed(causal, window, seg, t, kk)) continue;
          const double p = exp(s[kk] - l);
          const double ds = p * (dot_q_k(ob + (size_t)t * d, vb + (size_t)kk * d, d) - Dt);
          for (int c = 0; c < d; ++c) g[c] += scale * ds * widen_bf16(kb[(size_t)kk * d + c]);
        }
      } else {
        const long kk = krows[x - nq];
        double* gk = dk + ((size_t)bh * nk + (x - nq)) * d;
        double* gv = dv + ((size_t)bh * nk + (x - nq)) * d;
        for (int c = 0; c < d; ++c) gk[c] = gv[c] = 0.0;
        for (long t = 0; t < N; ++t) {
          if (!allowed(causal, window, seg, t, kk)) continue;
          double l, Dt;
          row_lse_and_D(qb + (size_t)t * d, ob + (size_t)t * d, t, kb, vb, N, d, causal, window, seg, scale, s, o,
                        &l, &Dt);
          const double p = exp(scale * dot_q_k(qb + (size_t)t * d, kb + (size_t)kk * d, d) - l);
          const double ds = p * (dot_q_k(ob + (size_t)t * d, vb + (size_t)kk * d, d) - Dt);
          for (int c = 0; c < d; ++c) {
            gk[c] += scale * ds * widen_bf16(qb[(size_t)t * d + c]);
            gv[c] += p * widen_bf16(ob[(size_t)t * d + c]);
          }
        }
      }
    }
    free(s);
    free(o);
  }
  return failed ? -2 : 0;
}

/*
 * dK and dV at sampled key positions from the forward's saved statistics
 * (the data the ring's backward also starts from: [RA-CN] "Backward
 * 需要让梯度也沿环传播" recomputes the probabilities from the saved logsumexp).
 * For key kk and every query t allowed to see it:
 *   D_t    = dO_t . out_t
 *   P_tk   = exp(scale q_t . k_kk - lse_t)
 *   dK_kk += scale P_tk (dO_t . v_kk - D_t) q_t
 *   dV_kk += P_tk dO_t
 * out [BH][N][d] and lse [BH][N] are doubles in natural order (the dense
 * forward's); dk, dv are [BH][nk][d].  With the exact out and lse this is
 * the plain definition of the two gradients; the cost per key is one pass
 * over its queries, so keys that every query sees stay cheap at any N.
 */
int oracle_dense_bwd_keys(int BH, long N, int d, int causal, long window, const long* seg, const uint16_t* q,
                          const uint16_t* k, const uint16_t* v, const uint16_t* dout, const double* out,
                          const double* lse, long nk, const long* krows, double* dk, double* dv, int nthreads) {
  if (BH <= 0 || N <= 0 || d <= 0 || nk < 0) return -1;
  set_threads(nthreads);
  const double scale = 1.0 / sqrt((double)d);
  const long total = (long)BH * nk;
#pragma omp parallel for schedule(dynamic, 1)
  for (long idx = 0; idx < total; ++idx) {
    const long bh = idx / nk, kk = krows[idx % nk];
    const uint16_t* qb = q + (size_t)bh * N * d;
    const uint16_t* ob = dout + (size_t)bh * N * d;
    const uint16_t* krow = k + ((size_t)bh * N + kk) * d;
    const uint16_t* vrow = v + ((size_t)bh * N + kk) * d;
    double* gk = dk + (size_t)idx * d;
    double* gv = dv + (size_t)idx * d;
    for (int c = 0; c < d; ++c) gk[c] = gv[c] = 0.0;
    for (long t = 0; t < N; ++t) {
      if (!allowed(causal, window, seg, t, kk)) continue;
      const uint16_t* qrow = qb + (size_t)t * d;
      const uint16_t* dorow = ob + (size_t)t * d;
      const double* orow = out + ((size_t)bh * N + t) * d;
      double Dt = 0.0;
      for (int c = 0; c < d; ++c) Dt += widen_bf16(dorow[c]) * orow[c];
      const double p = exp(scale * dot_q_k(qrow, krow, d) - lse[(size_t)bh * N + t]);
      const double ds = p * (dot_q_k(dorow, vrow, d) - Dt);
      for (int c = 0; c < d; ++c) {
        gk[c] += scale * ds * widen_bf16(qrow[c]);
        gv[c] += p * widen_bf16(dorow[c]);
      }
    }
  }
  return 0;
}

/*
 * Ring simulation of the backward ([RA-CN] "Backward 需要让梯度也沿环传播": the
 * owner of a query shard accumulates its dQ from every K/V block; the dK and
 * dV of a travelling block accumulate the contributions of each query owner
 * it passes and return to the block's owner at the end; the probabilities
 * are recomputed from the forward's saved logsumexp).
 * Inputs: q, k, v, dout (bf16 bit patterns) and the forward's out and lse
 * (doubles), all in natural order.  First D_t = dO_t . out_t for every row.
 * P virtual ranks; at step s rank r holds block j = (r - s) mod P together
 * with that block's accumulators (dK~, dV~); for its allowed pairs (i, k):
 *   P_ik = exp(scale q_i . k_k - lse_i),  dS_ik = P_ik (dO_i . v_k - D_i)
 *   dQ_i += scale dS_ik k_k   (kept by rank r)
 *   dK~_k += scale dS_ik q_i,  dV~_k += P_ik dO_i   (travel with block j)
 * then every rank passes block j and its accumulators to rank r + 1.  After
 * P steps each block's accumulators are back at its owner, which writes
 * them as dK, dV.  Outputs dq, dk, dv are [BH][N][d] doubles in natural
 * order; visits (NULL or [BH][N][N]) counts every (query, key) pair used.
 */
int oracle_ring_bwd(int BH, long N, int d, int P, int causal, long window, const long* seg, int layout,
                    const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout,
                    const double* out, const double* lse, double* dq, double* dk, double* dv,
                    long* visits, int nthreads) {
  if (BH <= 0 || N <= 0 || d <= 0 || !layout_ok(layout, N, P)) return -1;
  set_threads(nthreads);
  const long n = N / P;
  const double scale = 1.0 / sqrt((double)d);
  int failed = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int bh = 0; bh < BH; ++bh) {
    const size_t base = (size_t)bh * N;
    double* D = (double*)malloc(sizeof(double) * (size_t)N);
    /* accumulators by the rank holding them: acc[holder][local key][c] */
    double* accK = (double*)calloc((size_t)P * n * d, sizeof(double));
    double* accV = (double*)calloc((size_t)P * n * d, sizeof(double));
    double* nextK = (double*)malloc(sizeof(double) * (size_t)P * n * d);
    double* nextV = (double*)malloc(sizeof(double) * (size_t)P * n * d);
    if (!D || !accK || !accV || !nextK || !nextV) {
#pragma omp atomic write
      failed = 1;
      free(D); free(accK); free(accV); free(nextK); free(nextV);
      continue;
    }
    for (long t = 0; t < N; ++t) {
      double acc = 0.0;
      for (int c = 0; c < d; ++c) acc += widen_bf16(dout[(base + t) * d + c]) * out[(base + t) * d + c];
      D[t] = acc;
    }
    for (long t = 0; t < N; ++t)
      for (int c = 0; c < d; ++c) dq[(base + t) * d + c] = 0.0;
    for (int step = 0; step < P; ++step) {
      for (int r = 0; r < P; ++r) {
        const int j = oracle_block_at(P, r, step);
        double* aK = accK + (size_t)r * n * d;
        double* aV = accV + (size_t)r * n * d;
        for (long i = 0; i < n; ++i) {
          const long tq = oracle_position(layout, n, P, r, i);
          const uint16_t* qrow = q + (base + tq) * d;
          const uint16_t* dorow = dout + (base + tq) * d;
          double* g = dq + (base + tq) * d;
          for (long kk = 0; kk < n; ++kk) {
            const long tk = oracle_position(layout, n, P, j, kk);
            if (!allowed(causal, window, seg, tq, tk)) continue;
            const uint16_t* krow = k + (base + tk) * d;
            const uint16_t* vrow = v + (base + tk) * d;
            const double p = exp(scale * dot_q_k(qrow, krow, d) - lse[base + tq]);
            const double ds = p * (dot_q_k(dorow, vrow, d) - D[tq]);
            for (int c = 0; c < d; ++c) {
              g[c] += scale * ds * widen_bf16(krow[c]);
              aK[(size_t)kk * d + c] += scale * ds * widen_bf16(qrow[c]);
              aV[(size_t)kk * d + c] += p * widen_bf16(dorow[c]);
            }
            if (visits) visits[(base + tq) * N + tk] += 1;
          }
        }
      }
      /* rank r passes its block's accumulators to rank r + 1 */
      for (int r = 0; r < P; ++r) {
        const int to = (r + 1) % P;
        memcpy(nextK + (size_t)to * n * d, accK + (size_t)r * n * d, sizeof(double) * (size_t)n * d);
        memcpy(nextV + (size_t)to * n * d, accV + (size_t)r * n * d, sizeof(double) * (size_t)n * d);
      }
      double* tK = accK; accK = nextK; nextK = tK;
      double* tV = accV; accV = nextV; nextV = tV;
    }
    /* back at the owner: rank j holds block j's accumulators */
    for (int j = 0; j < P; ++j)
      for (long kk = 0; kk < n; ++kk) {
        const long tk = oracle_position(layout, n, P, j, kk);
        memcpy(dk + (base + tk) * d, accK + ((size_t)j * n + kk) * d, sizeof(double) * d);
        memcpy(dv + (base + tk) * d, accV + ((size_t)j * n + kk) * d, sizeof(double) * d);
      }
    free(D); free(accK); free(accV); free(nextK); free(nextV);
  }
  return failed ? -2 : 0;
}
