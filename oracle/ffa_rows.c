/* Row-by-row fp64 attention over AttnSlice masks, for checking sampled outputs
 * of large problems.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by tests/ (through oracle/rows_c.py) and
 * never by the library.  It shares no code with the CUDA path.
 *
 * It computes the same definitions as ffa_oracle.py (MagiAttention blog,
 * "Flex-Flash-Attention and AttnSlice": AttnSlice (QRange, KRange, MaskType),
 * the union of slices as the global mask; softmax attention and its analytic
 * gradients), one query row at a time and over the allowed keys only, so that
 * a row of a 1M-token problem costs its own key count and no dense block:
 *
 *   mask   key j is allowed to row i iff some slice (qs, qe, ks, ke, type)
 *          holds i in [qs, qe), j in [ks, ke) and, with r = i - qs,
 *          c = j - ks, Lq = qe - qs, Lk = ke - ks:
 *            FULL        always
 *            CAUSAL      c <= r + Lk - Lq        (bottom-right aligned)
 *            INV_CAUSAL  c >= r                  (top-left aligned)
 *            BI_CAUSAL   both
 *          For a fixed row each predicate is a bound on c, so a slice gives
 *          the row one interval of keys; the row's keys are their union.
 *   fwd    s_j = scale <q_i, k_j>; lse = ln sum_j exp(s_j); out = sum_j
 *          exp(s_j - lse) v_j; a row without keys: out 0, lse -inf.
 *   bwd    P_j = exp(s_j - lse), D = <dO_i, out_i>, dP_j = <dO_i, v_j>,
 *          dS_j = P_j (dP_j - D); dq_i = scale sum_j dS_j k_j;
 *          dk_j = scale sum_{h in group} sum_i dS_ij q_i, dv_j = sum_{h in
 *          group} sum_i P_ij dO_i.
 *   GQA    q head h uses kv head h / (hq / hkv).
 *
 * Inputs are bf16 bit patterns (widened exactly to double); every sum is in
 * double.  OpenMP splits the work over rows (forward, dq) or over keys
 * (dk, dv); each output element is summed by one thread.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { M_FULL = 0, M_CAUSAL = 1, M_INV_CAUSAL = 2, M_BI_CAUSAL = 3 };

typedef struct {
  int64_t lo, hi; /* [lo, hi) */
} ivl;

static double widen(uint16_t x) {
  uint32_t u = (uint32_t)x << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static void widen_row(const uint16_t* src, double* dst, int d) {
  for (int t = 0; t < d; ++t) dst[t] = widen(src[t]);
}

static double dot(const double* a, const double* b, int d) {
  double acc = 0.0;
#pragma omp simd reduction(+ : acc)
  for (int t = 0; t < d; ++t) acc += a[t] * b[t];
  return acc;
}

static int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }
static int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }

/* Keys of one slice allowed to row i, as an absolute [lo, hi) (empty: lo == hi). */
static void slice_row_keys(const int64_t* s, int64_t i, int64_t* lo, int64_t* hi) {
  const int64_t qs = s[0], qe = s[1], ks = s[2], ke = s[3], type = s[4];
  *lo = *hi = 0;
  if (i < qs || i >= qe || ke <= ks) return;
  const int64_t r = i - qs, lq = qe - qs, lk = ke - ks;
  int64_t c0 = 0, c1 = lk; /* local [c0, c1) */
  if (type == M_CAUSAL || type == M_BI_CAUSAL) c1 = min64(c1, r + lk - lq + 1);
  if (type == M_INV_CAUSAL || type == M_BI_CAUSAL) c0 = max64(c0, r);
  if (c1 <= c0) return;
  *lo = ks + c0;
  *hi = ks + c1;
}

static int cmp_ivl(const void* a, const void* b) {
  const ivl* x = (const ivl*)a;
  const ivl* y = (const ivl*)b;
  return x->lo < y->lo ? -1 : (x->lo > y->lo ? 1 : 0);
}

/* Allowed keys of row i: the union of the slices' intervals (clipped to
 * [0, sk)), sorted and merged.  ivs holds n_slices entries; returns the count. */
static int64_t row_keys(const int64_t* slices, int64_t ns, int64_t i, int64_t sk, ivl* ivs) {
  int64_t n = 0;
  for (int64_t s = 0; s < ns; ++s) {
    int64_t lo, hi;
    slice_row_keys(slices + 5 * s, i, &lo, &hi);
    lo = max64(lo, 0);
    hi = min64(hi, sk);
    if (hi > lo) ivs[n++] = (ivl){lo, hi};
  }
  qsort(ivs, (size_t)n, sizeof(ivl), cmp_ivl);
  int64_t m = 0;
  for (int64_t x = 0; x < n; ++x) {
    if (m > 0 && ivs[x].lo <= ivs[m - 1].hi) {
      ivs[m - 1].hi = max64(ivs[m - 1].hi, ivs[x].hi);
    } else {
      ivs[m++] = ivs[x];
    }
  }
  return m;
}

static int64_t count_keys(const ivl* ivs, int64_t n) {
  int64_t c = 0;
  for (int64_t x = 0; x < n; ++x) c += ivs[x].hi - ivs[x].lo;
  return c;
}

static int args_ok(int64_t sq, int64_t sk, int32_t hq, int32_t hkv, int32_t d, int64_t ns) {
  return sq >= 0 && sk >= 0 && hq > 0 && hkv > 0 && hq % hkv == 0 && d > 0 && ns >= 0;
}

/* out [nr][hq][d], lse [hq][nr] and, when dout and dq are given, dq
 * [nr][hq][d] of the listed rows.  Returns 0, or 1 on bad arguments, 2 when
 * memory runs out. */
int ffa_oracle_rows(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout, int64_t sq,
                    int64_t sk, int32_t hq, int32_t hkv, int32_t d, const int64_t* slices, int64_t ns, double scale,
                    const int64_t* rows, int64_t nr, double* out, double* lse, double* dq) {
  if (!args_ok(sq, sk, hq, hkv, d, ns)) return 1;
  for (int64_t x = 0; x < nr; ++x)
    if (rows[x] < 0 || rows[x] >= sq) return 1;
  const int G = hq / hkv;
  const int grad = dout != NULL && dq != NULL;
  /* the longest row decides the per-thread score buffers */
  int64_t maxkeys = 0;
  int fail = 0;
#pragma omp parallel reduction(max : maxkeys) reduction(| : fail)
  {
    ivl* ivs = (ivl*)malloc(sizeof(ivl) * (size_t)(ns + 1));
    if (!ivs) {
      fail = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t x = 0; x < nr; ++x) maxkeys = max64(maxkeys, count_keys(ivs, row_keys(slices, ns, rows[x], sk, ivs)));
      free(ivs);
    }
  }
  if (fail) return 2;
#pragma omp parallel reduction(| : fail)
  {
    ivl* ivs = (ivl*)malloc(sizeof(ivl) * (size_t)(ns + 1));
    /* per allowed key (in order) and head: s, then exp(s - max), then P; and dP */
    double* e = (double*)malloc(sizeof(double) * (size_t)(hq * maxkeys + 1));
    double* dp = (double*)malloc(sizeof(double) * (size_t)(hq * maxkeys + 1));
    double* kd = (double*)malloc(sizeof(double) * (size_t)(hkv * d));          /* k_j or v_j, every kv head */
    double* qd = (double*)malloc(sizeof(double) * (size_t)(hq * d));
    double* od = (double*)malloc(sizeof(double) * (size_t)(hq * d));
    double* dod = (double*)malloc(sizeof(double) * (size_t)(hq * d));
    double* dqd = (double*)malloc(sizeof(double) * (size_t)(hq * d));
    double* mx = (double*)malloc(sizeof(double) * (size_t)hq);
    double* dd = (double*)malloc(sizeof(double) * (size_t)hq);
    if (!ivs || !e || !dp || !kd || !qd || !od || !dod || !dqd || !mx || !dd) {
      fail = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t x = 0; x < nr; ++x) {
        const int64_t i = rows[x];
        const int64_t niv = row_keys(slices, ns, i, sk, ivs);
        const int64_t n = count_keys(ivs, niv);
        if (n == 0) { /* no allowed key: out 0, lse -inf, dq 0 */
          for (int h = 0; h < hq; ++h) lse[(int64_t)h * nr + x] = -INFINITY;
          memset(out + x * hq * (int64_t)d, 0, sizeof(double) * (size_t)(hq * d));
          if (grad) memset(dq + x * hq * (int64_t)d, 0, sizeof(double) * (size_t)(hq * d));
          continue;
        }
        widen_row(q + i * hq * (int64_t)d, qd, hq * d);
        if (grad) widen_row(dout + i * hq * (int64_t)d, dod, hq * d);
        for (int h = 0; h < hq; ++h) mx[h] = -INFINITY;
        /* pass 1: scores s_j of every head and their maxima */
        int64_t c = 0;
        for (int64_t a = 0; a < niv; ++a)
          for (int64_t j = ivs[a].lo; j < ivs[a].hi; ++j, ++c) {
            widen_row(k + j * hkv * (int64_t)d, kd, hkv * d);
            for (int h = 0; h < hq; ++h) {
              const double s = scale * dot(qd + h * d, kd + (h / G) * d, d);
              e[c * hq + h] = s;
              if (s > mx[h]) mx[h] = s;
            }
          }
        /* lse = max + ln sum exp(s - max); P_j = exp(s_j - max) / sum */
        for (int h = 0; h < hq; ++h) dd[h] = 0.0;   /* the sums */
        for (int64_t j = 0; j < n; ++j)
          for (int h = 0; h < hq; ++h) {
            e[j * hq + h] = exp(e[j * hq + h] - mx[h]);
            dd[h] += e[j * hq + h];
          }
        for (int h = 0; h < hq; ++h) lse[(int64_t)h * nr + x] = mx[h] + log(dd[h]);
        for (int64_t j = 0; j < n; ++j)
          for (int h = 0; h < hq; ++h) e[j * hq + h] /= dd[h];
        /* pass 2: out = sum_j P_j v_j and dP_j = <dO, v_j> */
        memset(od, 0, sizeof(double) * (size_t)(hq * d));
        c = 0;
        for (int64_t a = 0; a < niv; ++a)
          for (int64_t j = ivs[a].lo; j < ivs[a].hi; ++j, ++c) {
            widen_row(v + j * hkv * (int64_t)d, kd, hkv * d);
            for (int h = 0; h < hq; ++h) {
              const double p = e[c * hq + h];
              const double* vg = kd + (h / G) * d;
              double* o = od + h * d;
              for (int t = 0; t < d; ++t) o[t] += p * vg[t];
              if (grad) dp[c * hq + h] = dot(dod + h * d, vg, d);
            }
          }
        memcpy(out + x * hq * (int64_t)d, od, sizeof(double) * (size_t)(hq * d));
        if (!grad) continue;
        /* pass 3: dq = scale sum_j P_j (dP_j - D) k_j, D = <dO, out> */
        for (int h = 0; h < hq; ++h) dd[h] = dot(dod + h * d, od + h * d, d);
        memset(dqd, 0, sizeof(double) * (size_t)(hq * d));
        c = 0;
        for (int64_t a = 0; a < niv; ++a)
          for (int64_t j = ivs[a].lo; j < ivs[a].hi; ++j, ++c) {
            widen_row(k + j * hkv * (int64_t)d, kd, hkv * d);
            for (int h = 0; h < hq; ++h) {
              const double ds = e[c * hq + h] * (dp[c * hq + h] - dd[h]);
              const double* kg = kd + (h / G) * d;
              double* r = dqd + h * d;
              for (int t = 0; t < d; ++t) r[t] += ds * kg[t];
            }
          }
        double* r = dq + x * hq * (int64_t)d;
        for (int t = 0; t < hq * d; ++t) r[t] = scale * dqd[t];
      }
    }
    free(ivs);
    free(e);
    free(dp);
    free(kd);
    free(qd);
    free(od);
    free(dod);
    free(dqd);
    free(mx);
    free(dd);
  }
  return fail ? 2 : 0;
}

/* Is key j inside one of the sorted intervals ivs[0..n)? */
static int key_in(const ivl* ivs, int64_t n, int64_t j) {
  int64_t lo = 0, hi = n;
  while (lo < hi) {
    const int64_t mid = (lo + hi) / 2;
    if (ivs[mid].hi <= j) lo = mid + 1;
    else hi = mid;
  }
  return lo < n && ivs[lo].lo <= j;
}

/* Does the row's key set meet the sorted key list? */
static int meets(const ivl* ivs, int64_t n, const int64_t* keys, int64_t nk) {
  for (int64_t a = 0; a < n; ++a) {
    int64_t lo = 0, hi = nk; /* first key >= ivs[a].lo */
    while (lo < hi) {
      const int64_t mid = (lo + hi) / 2;
      if (keys[mid] < ivs[a].lo) lo = mid + 1;
      else hi = mid;
    }
    if (lo < nk && keys[lo] < ivs[a].hi) return 1;
  }
  return 0;
}

/* dk, dv [nk][hkv][d] of the listed keys (sorted ascending, distinct): the
 * sums over every row allowed to the key and every q head of its group.
 * Returns 0, 1 on bad arguments, 2 when memory runs out. */
int ffa_oracle_keys(const uint16_t* q, const uint16_t* k, const uint16_t* v, const uint16_t* dout, int64_t sq,
                    int64_t sk, int32_t hq, int32_t hkv, int32_t d, const int64_t* slices, int64_t ns, double scale,
                    const int64_t* keys, int64_t nk, double* dk, double* dv) {
  if (!args_ok(sq, sk, hq, hkv, d, ns)) return 1;
  for (int64_t x = 0; x < nk; ++x)
    if (keys[x] < 0 || keys[x] >= sk || (x > 0 && keys[x] <= keys[x - 1])) return 1;
  memset(dk, 0, sizeof(double) * (size_t)(nk * hkv * d));
  memset(dv, 0, sizeof(double) * (size_t)(nk * hkv * d));
  if (nk == 0 || sq == 0) return 0;
  const int G = hq / hkv;
  /* 1. the rows allowed to at least one listed key */
  char* use = (char*)calloc((size_t)sq, 1);
  if (!use) return 2;
  int fail = 0;
#pragma omp parallel reduction(| : fail)
  {
    ivl* ivs = (ivl*)malloc(sizeof(ivl) * (size_t)(ns + 1));
    if (!ivs) {
      fail = 1;
    } else {
#pragma omp for schedule(static)
      for (int64_t i = 0; i < sq; ++i) use[i] = (char)meets(ivs, row_keys(slices, ns, i, sk, ivs), keys, nk);
    }
    free(ivs);
  }
  int64_t nr = 0;
  for (int64_t i = 0; i < sq; ++i) nr += use[i];
  int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nr + 1));
  int64_t* ivoff = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nr + 1));
  ivl* rivs = (ivl*)malloc(sizeof(ivl) * (size_t)(nr * (ns + 1) + 1));
  double* out = (double*)malloc(sizeof(double) * (size_t)(nr * hq * d + 1));
  double* lse = (double*)malloc(sizeof(double) * (size_t)(nr * hq + 1));
  double* D = (double*)malloc(sizeof(double) * (size_t)(nr * hq + 1));
  if (fail || !rows || !ivoff || !rivs || !out || !lse || !D) {
    free(use), free(rows), free(ivoff), free(rivs), free(out), free(lse), free(D);
    return 2;
  }
  nr = 0;
  for (int64_t i = 0; i < sq; ++i)
    if (use[i]) rows[nr++] = i;
  free(use);
  /* 2. their forward (lse, out), D = <dO, out>, and their key intervals */
  int rc = ffa_oracle_rows(q, k, v, NULL, sq, sk, hq, hkv, d, slices, ns, scale, rows, nr, out, lse, NULL);
  if (rc != 0) {
    free(rows), free(ivoff), free(rivs), free(out), free(lse), free(D);
    return rc;
  }
#pragma omp parallel for schedule(static)
  for (int64_t x = 0; x < nr; ++x) {
    ivoff[x] = row_keys(slices, ns, rows[x], sk, rivs + x * (ns + 1));
    for (int h = 0; h < hq; ++h) {
      double s = 0.0;
      for (int t = 0; t < d; ++t)
        s += widen(dout[((rows[x] * hq) + h) * (int64_t)d + t]) * out[((x * hq) + h) * (int64_t)d + t];
      D[x * hq + h] = s;
    }
  }
  free(out);
  /* 3. per key: dv_j = sum P_ij dO_i, dk_j = scale sum dS_ij q_i over the allowed rows and the group's heads */
#pragma omp parallel reduction(| : fail)
  {
    double* kd = (double*)malloc(sizeof(double) * (size_t)(hkv * d));
    double* vd = (double*)malloc(sizeof(double) * (size_t)(hkv * d));
    double* qd = (double*)malloc(sizeof(double) * (size_t)(hq * d));
    double* dod = (double*)malloc(sizeof(double) * (size_t)(hq * d));
    if (!kd || !vd || !qd || !dod) {
      fail = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t y = 0; y < nk; ++y) {
        const int64_t j = keys[y];
        widen_row(k + j * hkv * (int64_t)d, kd, hkv * d);
        widen_row(v + j * hkv * (int64_t)d, vd, hkv * d);
        for (int64_t x = 0; x < nr; ++x) {
          if (!key_in(rivs + x * (ns + 1), ivoff[x], j)) continue;
          const int64_t i = rows[x];
          widen_row(q + i * hq * (int64_t)d, qd, hq * d);
          widen_row(dout + i * hq * (int64_t)d, dod, hq * d);
          for (int h = 0; h < hq; ++h) {
            const int g = h / G;
            double* rk = dk + ((y * hkv) + g) * (int64_t)d;
            double* rv = dv + ((y * hkv) + g) * (int64_t)d;
            const double* qh = qd + h * d;
            const double* doh = dod + h * d;
            const double p = exp(scale * dot(qh, kd + g * d, d) - lse[h * nr + x]);
            const double ds = p * (dot(doh, vd + g * d, d) - D[x * hq + h]);
            for (int t = 0; t < d; ++t) {
              rv[t] += p * doh[t];
              rk[t] += scale * ds * qh[t];
            }
          }
        }
      }
    }
    free(kd);
    free(vd);
    free(qd);
    free(dod);
  }
  free(rows), free(ivoff), free(rivs), free(lse), free(D);
  return fail ? 2 : 0;
}
