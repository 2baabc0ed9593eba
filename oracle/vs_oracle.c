/*
 * vs_oracle.c -- plain, slow, fp64 CPU reference for MTraining's dynamic
 * Vertical-Slash (VS) sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the package's smoke check and the
 * benchmark's CPU-baseline leg do.
 *
 * It shares no code, header, table or constant with the CUDA library.
 * Inputs are double arrays (exact bf16 values when they come from the
 * generator); every product and sum is formed in double.
 *
 * Sources (MTraining: Distributed Dynamic Sparse Attention for Efficient
 * Ultra-Long Context Training):
 *   - Vertical-Slash pattern: a slash is a diagonal n-m = const, a vertical a
 *     key column m (section 3.2).
 *   - Algorithm 1 (Dynamic sparse training head): A_hat = softmax(Q[-last_q:]
 *     K^T / sqrt(d) + causal mask); sum_v(A_hat) per key column; sum_s(A_hat)
 *     per diagonal; argtopk of each.
 *   - Eq. 1: dL/dS = A (.) (dL/dA - rowsum(dL/dA (.) A)).
 *   - Eq. 2 (appendix B.1): dL/dV = A^T dL/dO; dL/dQ = (1/sqrt d) dL/dS K;
 *     dL/dK = (1/sqrt d) (dL/dS)^T Q.
 *   - Algorithm 2 (Hierarchical Balanced Sparse Ring Attention):
 *     merge_out_and_lse of partial (Out, LSE) results.
 *   - Section 4.2 (ii): block-level striping with 64-token stripes.
 *
 * Readings taken where the pages are silent (listed again in the design
 * notes): budgets are fixed top-k; the mask is the exact token-level union
 * M[n,m] = (m <= n) and (m in iv or n-m in is); a row with an empty mask has
 * O = 0, LSE = -inf and no gradient; ties in top-k go to the lower index; the
 * KV head of query head h is h / (Hq/Hkv); dK and dV of a KV head are summed
 * over its query heads.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Problem description.  Tensors are token-major: x[b][n][h][c]. */
typedef struct {
  int B, Nq, Nk, Hq, Hkv, d;
  int64_t n_global;      /* length of the global sequence (index space of iv/is) */
  const double* q;        /* [B][Nq][Hq][d] */
  const double* k;        /* [B][Nk][Hkv][d] */
  const double* v;        /* [B][Nk][Hkv][d] */
  const double* dout;     /* [B][Nq][Hq][d] or NULL (forward only) */
  const int64_t* qpos;   /* [Nq] global position of each local query row */
  const int64_t* kpos;   /* [Nk] global position of each local key */
  const int32_t* iv;     /* [B][Hq][kv] selected key columns (global) */
  const int32_t* is;     /* [B][Hq][ks] selected offsets n-m */
  int kv, ks;
  double scale;
  int block; /* 0: the exact token mask; 1: block-cover slashes (see mask_row) */
} ora_problem;

int ora_version(void) { return 4; }

int ora_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ top-k */
/* Total order used for selection: larger score first, then lower index. */
typedef struct {
  double s;
  int32_t i;
} scored;

static int cmp_desc_score_then_index(const void* a, const void* b) {
  const scored* x = (const scored*)a;
  const scored* y = (const scored*)b;
  if (x->s > y->s) return -1;
  if (x->s < y->s) return 1;
  return (x->i < y->i) ? -1 : (x->i > y->i);
}
static int cmp_i32(const void* a, const void* b) {
  int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
  return (x < y) ? -1 : (x > y);
}

/* argtopk (Algorithm 1): the k indices with the largest scores under the
 * total order above, returned sorted ascending. */
void ora_topk(int n, const double* score, int k, int32_t* out) {
  scored* t = (scored*)malloc(sizeof(scored) * (size_t)n);
  for (int i = 0; i < n; ++i) {
    t[i].s = score[i];
    t[i].i = i;
  }
  qsort(t, (size_t)n, sizeof(scored), cmp_desc_score_then_index);
  for (int j = 0; j < k; ++j) out[j] = t[j].i;
  qsort(out, (size_t)k, sizeof(int32_t), cmp_i32);
  free(t);
}

/* ------------------------------------------------------------- estimator */
/* Algorithm 1, first four lines, for every (b, h):
 *   rows n_i = N - last_q + i, i in [0, last_q);
 *   A_hat[i, m] = softmax over m <= n_i of scale * q_{n_i} . k_m;
 *   v[m] = sum_i A_hat[i, m];   s[o] = sum_i A_hat[i, n_i - o].
 * Outputs v, s: [B][Hq][N]. */
void ora_estimate(int B, int N, int Hq, int Hkv, int d, const double* q, const double* k, int last_q, double scale,
                  double* vout, double* sout) {
  const int g = Hq / Hkv;
#pragma omp parallel for collapse(2) schedule(dynamic)
  for (int b = 0; b < B; ++b)
    for (int h = 0; h < Hq; ++h) {
      const int hk = h / g;
      double* vs = vout + ((size_t)b * Hq + h) * N;
      double* ss = sout + ((size_t)b * Hq + h) * N;
      double* logit = (double*)malloc(sizeof(double) * (size_t)N);
      for (int m = 0; m < N; ++m) vs[m] = ss[m] = 0.0;
      for (int i = 0; i < last_q; ++i) {
        const int n = N - last_q + i;
        const double* qn = q + (((size_t)b * N + n) * Hq + h) * d;
        double mx = -INFINITY;
        for (int m = 0; m <= n; ++m) {
          const double* km = k + (((size_t)b * N + m) * Hkv + hk) * d;
          double dot = 0.0;
          for (int c = 0; c < d; ++c) dot += (double)qn[c] * (double)km[c];
          logit[m] = scale * dot;
          if (logit[m] > mx) mx = logit[m];
        }
        double z = 0.0;
        for (int m = 0; m <= n; ++m) z += exp(logit[m] - mx);
        for (int m = 0; m <= n; ++m) {
          const double a = exp(logit[m] - mx) / z;
          vs[m] += a;        /* vertical: column m */
          ss[n - m] += a;    /* slash: diagonal o = n - m */
        }
      }
      free(logit);
    }
}

/* ------------------------------------------------------------- the mask */
/* Per (b, h) membership tables over the global index space. */
typedef struct {
  unsigned char* vsel; /* vsel[c] = 1 iff c in iv */
  unsigned char* ssel; /* ssel[o] = 1 iff o in is */
  unsigned char* bact; /* block mode: bact[D] = 1 iff a selected slash passes through a 64x64 block of block diagonal D */
  int64_t* loc;        /* global key position -> local key index, or -1 */
} ora_tables;

static void tables_build(const ora_problem* p, int b, int h, ora_tables* t) {
  const int64_t G = p->n_global;
  t->vsel = (unsigned char*)calloc((size_t)G, 1);
  t->ssel = (unsigned char*)calloc((size_t)G, 1);
  t->loc = (int64_t*)malloc(sizeof(int64_t) * (size_t)G);
  for (int64_t x = 0; x < G; ++x) t->loc[x] = -1;
  for (int m = 0; m < p->Nk; ++m) t->loc[p->kpos[m]] = m;
  const int32_t* iv = p->iv + ((size_t)b * p->Hq + h) * p->kv;
  const int32_t* is = p->is + ((size_t)b * p->Hq + h) * p->ks;
  /* entries < 0 pad a list whose budget is below its capacity (top-p) */
  for (int j = 0; j < p->kv; ++j)
    if (iv[j] >= 0) t->vsel[iv[j]] = 1;
  for (int j = 0; j < p->ks; ++j)
    if (is[j] >= 0) t->ssel[is[j]] = 1;
  /* block diagonal D holds the blocks (I, I - D); the slash at offset o
   * passes through one of them iff some n - m = o with n, m in blocks I and
   * I - D, i.e. iff |o - 64 D| <= 63 */
  const int64_t nd = G / 64 + 1;
  t->bact = (unsigned char*)calloc((size_t)nd, 1);
  for (int64_t D = 0; D < nd; ++D)
    for (int64_t o = 64 * D - 63; o <= 64 * D + 63; ++o)
      if (o >= 0 && o < G && t->ssel[o]) {
        t->bact[D] = 1;
        break;
      }
}
static void tables_free(ora_tables* t) {
  free(t->vsel);
  free(t->ssel);
  free(t->bact);
  free(t->loc);
}

/* Membership of the key at global position pm in the mask row of the query
 * at global position pn (the same rule mask_row enumerates). */
static int in_mask(const ora_problem* p, const ora_tables* t, int64_t pn, int64_t pm) {
  if (pm > pn) return 0;
  if (t->vsel[pm]) return 1;
  return p->block ? t->bact[(pn >> 6) - (pm >> 6)] : t->ssel[pn - pm];
}

/* Capacity of a row's key list: distinct keys, at most one per list entry
 * (exact mask) or any key (block cover). */
static size_t row_cap(const ora_problem* p) {
  const int64_t lists = (int64_t)p->kv + p->ks;
  return (size_t)((p->block || lists > p->Nk ? p->Nk : lists) + 1);
}

/* Enumerates M(n) for local query row n: local key indices m with
 * kpos[m] <= qpos[n] and (kpos[m] in iv or qpos[n] - kpos[m] in is).
 * Each key appears once.  Returns the count; keys written to `out`. */
static int mask_row(const ora_problem* p, int b, int h, const ora_tables* t, int n, int32_t* out) {
  const int64_t pn = p->qpos[n];
  const int32_t* iv = p->iv + ((size_t)b * p->Hq + h) * p->kv;
  const int32_t* is = p->is + ((size_t)b * p->Hq + h) * p->ks;
  int cnt = 0;
  if (p->block) {
    /* block cover: every causal entry of a 64x64 block that a selected slash
     * passes through, plus the selected columns */
    for (int m = 0; m < p->Nk; ++m) {
      const int64_t pm = p->kpos[m];
      if (pm > pn) continue;
      if (t->vsel[pm] || t->bact[(pn >> 6) - (pm >> 6)]) out[cnt++] = m;
    }
    return cnt;
  }
  for (int j = 0; j < p->ks; ++j) { /* slash entries */
    if (is[j] < 0) continue;
    const int64_t pm = pn - is[j];
    if (pm < 0) continue;
    const int64_t m = t->loc[pm];
    if (m >= 0) out[cnt++] = (int32_t)m;
  }
  for (int j = 0; j < p->kv; ++j) { /* vertical entries not already on a selected diagonal */
    if (iv[j] < 0) continue;
    const int64_t pm = iv[j];
    if (pm > pn || t->ssel[pn - pm]) continue;
    const int64_t m = t->loc[pm];
    if (m >= 0) out[cnt++] = (int32_t)m;
  }
  return cnt;
}

/* Number of mask entries |M| summed over all (b, h, n): the effective mask
 * area that FLOPs are counted on. */
int64_t ora_mask_count(const ora_problem* p) {
  int64_t total = 0;
  for (int b = 0; b < p->B; ++b)
    for (int h = 0; h < p->Hq; ++h) {
      ora_tables t;
      tables_build(p, b, h, &t);
      int64_t part = 0;
#pragma omp parallel
      {
        int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * row_cap(p));
#pragma omp for reduction(+ : part) schedule(static)
        for (int n = 0; n < p->Nq; ++n) part += mask_row(p, b, h, &t, n, keys);
        free(keys);
      }
      total += part;
      tables_free(&t);
    }
  return total;
}

/* Writes the dense boolean mask of one head, [Nq][Nk] (small cases only). */
void ora_mask_dense(const ora_problem* p, int b, int h, unsigned char* out) {
  ora_tables t;
  tables_build(p, b, h, &t);
  int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * row_cap(p));
  memset(out, 0, (size_t)p->Nq * p->Nk);
  for (int n = 0; n < p->Nq; ++n) {
    int c = mask_row(p, b, h, &t, n, keys);
    for (int j = 0; j < c; ++j) out[(size_t)n * p->Nk + keys[j]] = 1;
  }
  free(keys);
  tables_free(&t);
}

static inline double dotd(const double* a, const double* b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

/* Row statistics of one query row: LSE_n = log sum_{m in M(n)} exp(S_nm)
 * and (when dout is given) D_n = sum_m dA_nm A_nm with dA = dO V^T (Eq. 1's
 * row sum).  Empty rows: LSE = -inf, D = 0. */
static void row_stats(const ora_problem* p, int b, int h, const ora_tables* t, int n, int32_t* keys,
                      double* logit, double* lse_out, double* D_out) {
  const int d = p->d, hk = h / (p->Hq / p->Hkv);
  const double* qn = p->q + (((size_t)b * p->Nq + n) * p->Hq + h) * d;
  const int c = mask_row(p, b, h, t, n, keys);
  if (c == 0) {
    *lse_out = -INFINITY;
    if (D_out) *D_out = 0.0;
    return;
  }
  double mx = -INFINITY;
  for (int j = 0; j < c; ++j) {
    const double* km = p->k + (((size_t)b * p->Nk + keys[j]) * p->Hkv + hk) * d;
    logit[j] = p->scale * dotd(qn, km, d);
    if (logit[j] > mx) mx = logit[j];
  }
  double z = 0.0;
  for (int j = 0; j < c; ++j) z += exp(logit[j] - mx);
  const double lse = mx + log(z);
  *lse_out = lse;
  if (D_out) {
    const double* don = p->dout + (((size_t)b * p->Nq + n) * p->Hq + h) * d;
    double D = 0.0;
    for (int j = 0; j < c; ++j) {
      const double* vm = p->v + (((size_t)b * p->Nk + keys[j]) * p->Hkv + hk) * d;
      D += dotd(don, vm, d) * exp(logit[j] - lse);
    }
    *D_out = D;
  }
}

/* LSE_n and D_n (Eq. 1's row sum of dA (.) A) for a list of (b, h, n) rows. */
void ora_row_stats(const ora_problem* p, int nrows, const int32_t* rows, double* lse, double* D) {
  for (int r = 0; r < nrows; ++r) {
    const int b = rows[3 * r], h = rows[3 * r + 1], n = rows[3 * r + 2];
    ora_tables t;
    tables_build(p, b, h, &t);
    int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * row_cap(p));
    double* logit = (double*)malloc(sizeof(double) * row_cap(p));
    row_stats(p, b, h, &t, n, keys, logit, &lse[r], p->dout ? &D[r] : NULL);
    free(keys);
    free(logit);
    tables_free(&t);
  }
}

/* Forward and the query-side backward for a list of rows.
 *   rows: nrows triples (b, h, n).
 *   o [nrows][d], lse [nrows]; dq [nrows][d] when p->dout != NULL (else may be NULL).
 * O_n = sum_m A_nm v_m; dQ_n = scale * sum_m dS_nm k_m with
 * dS_nm = A_nm (dA_nm - D_n) (Eq. 1, Eq. 2). */
void ora_rows(const ora_problem* p, int nrows, const int32_t* rows, double* o, double* lse, double* dq) {
  const int d = p->d;
  /* group rows by (b, h) so each head's tables are built once */
  for (int b = 0; b < p->B; ++b)
    for (int h = 0; h < p->Hq; ++h) {
      int any = 0;
      for (int r = 0; r < nrows && !any; ++r) any = (rows[3 * r] == b && rows[3 * r + 1] == h);
      if (!any) continue;
      ora_tables t;
      tables_build(p, b, h, &t);
      const int hk = h / (p->Hq / p->Hkv);
#pragma omp parallel
      {
        int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * row_cap(p));
        double* logit = (double*)malloc(sizeof(double) * row_cap(p));
#pragma omp for schedule(dynamic, 16)
        for (int r = 0; r < nrows; ++r) {
          if (rows[3 * r] != b || rows[3 * r + 1] != h) continue;
          const int n = rows[3 * r + 2];
          double L, D = 0.0;
          row_stats(p, b, h, &t, n, keys, logit, &L, p->dout ? &D : NULL);
          lse[r] = L;
          double* orow = o + (size_t)r * d;
          for (int c = 0; c < d; ++c) orow[c] = 0.0;
          if (dq)
            for (int c = 0; c < d; ++c) dq[(size_t)r * d + c] = 0.0;
          if (isinf(L)) continue;
          const int cnt = mask_row(p, b, h, &t, n, keys);
          const double* qn = p->q + (((size_t)b * p->Nq + n) * p->Hq + h) * d;
          const double* don = p->dout ? p->dout + (((size_t)b * p->Nq + n) * p->Hq + h) * d : NULL;
          for (int j = 0; j < cnt; ++j) {
            const double* km = p->k + (((size_t)b * p->Nk + keys[j]) * p->Hkv + hk) * d;
            const double* vm = p->v + (((size_t)b * p->Nk + keys[j]) * p->Hkv + hk) * d;
            const double A = exp(p->scale * dotd(qn, km, d) - L);
            for (int c = 0; c < d; ++c) orow[c] += A * (double)vm[c];
            if (dq && don) {
              const double dS = A * (dotd(don, vm, d) - D);
              for (int c = 0; c < d; ++c) dq[(size_t)r * d + c] += p->scale * dS * (double)km[c];
            }
          }
        }
        free(keys);
        free(logit);
      }
      tables_free(&t);
    }
}

/* Key-side backward for a list of keys.
 *   keys: nkeys triples (b, hk, m) with m a local key index.
 *   dk, dv [nkeys][d].
 * dV_m = sum_{h in group} sum_n A_nm dO_n;  dK_m = scale * sum_h sum_n dS_nm q_n.
 * Needs LSE_n and D_n of every row of the group's heads. */
void ora_keys(const ora_problem* p, int nkeys, const int32_t* keys_in, double* dk, double* dv) {
  const int d = p->d, g = p->Hq / p->Hkv;
  for (int r = 0; r < nkeys; ++r)
    for (int c = 0; c < d; ++c) dk[(size_t)r * d + c] = dv[(size_t)r * d + c] = 0.0;
  double* L = (double*)malloc(sizeof(double) * (size_t)p->Nq);
  double* D = (double*)malloc(sizeof(double) * (size_t)p->Nq);
  for (int b = 0; b < p->B; ++b)
    for (int hk = 0; hk < p->Hkv; ++hk) {
      int any = 0;
      for (int r = 0; r < nkeys && !any; ++r) any = (keys_in[3 * r] == b && keys_in[3 * r + 1] == hk);
      if (!any) continue;
      for (int h = hk * g; h < (hk + 1) * g; ++h) {
        ora_tables t;
        tables_build(p, b, h, &t);
#pragma omp parallel
        {
          int32_t* keys = (int32_t*)malloc(sizeof(int32_t) * row_cap(p));
          double* logit = (double*)malloc(sizeof(double) * row_cap(p));
#pragma omp for schedule(dynamic, 64)
          for (int n = 0; n < p->Nq; ++n) row_stats(p, b, h, &t, n, keys, logit, &L[n], &D[n]);
          free(keys);
          free(logit);
        }
        /* membership of key m in row n's mask (in_mask) */
#pragma omp parallel for schedule(dynamic, 1)
        for (int r = 0; r < nkeys; ++r) {
          if (keys_in[3 * r] != b || keys_in[3 * r + 1] != hk) continue;
          const int m = keys_in[3 * r + 2];
          const int64_t pm = p->kpos[m];
          const double* km = p->k + (((size_t)b * p->Nk + m) * p->Hkv + hk) * d;
          const double* vm = p->v + (((size_t)b * p->Nk + m) * p->Hkv + hk) * d;
          for (int n = 0; n < p->Nq; ++n) {
            const int64_t pn = p->qpos[n];
            if (!in_mask(p, &t, pn, pm)) continue;
            const double* qn = p->q + (((size_t)b * p->Nq + n) * p->Hq + h) * d;
            const double* don = p->dout + (((size_t)b * p->Nq + n) * p->Hq + h) * d;
            const double A = exp(p->scale * dotd(qn, km, d) - L[n]);
            const double dS = A * (dotd(don, vm, d) - D[n]);
            for (int c = 0; c < d; ++c) {
              dv[(size_t)r * d + c] += A * (double)don[c];
              dk[(size_t)r * d + c] += p->scale * dS * (double)qn[c];
            }
          }
        }
        tables_free(&t);
      }
    }
  free(L);
  free(D);
}

/* ------------------------------------------------- striping and merging */
/* Block-level striping (section 4.2 (ii)): global block j (of `stripe`
 * tokens) goes to worker j mod W at local block floor(j / W).  Writes the
 * global position of every local token of worker r: pos[N/W]. */
void ora_stripe_positions(int64_t N, int W, int stripe, int r, int64_t* pos) {
  const int64_t nloc = N / W;
  for (int64_t l = 0; l < nloc; ++l) {
    const int64_t jl = l / stripe, a = l % stripe;
    pos[l] = (jl * W + r) * stripe + a;
  }
}

/* merge_out_and_lse (Algorithm 2) for one row of width d:
 * LSE = log(e^L1 + e^L2), O = (e^L1 O1 + e^L2 O2) / e^LSE. */
void ora_merge(int d, const double* o1, double l1, const double* o2, double l2, double* o, double* l) {
  if (isinf(l1) && l1 < 0) {
    for (int c = 0; c < d; ++c) o[c] = o2[c];
    *l = l2;
    return;
  }
  if (isinf(l2) && l2 < 0) {
    for (int c = 0; c < d; ++c) o[c] = o1[c];
    *l = l1;
    return;
  }
  const double mx = l1 > l2 ? l1 : l2;
  const double lse = mx + log(exp(l1 - mx) + exp(l2 - mx));
  for (int c = 0; c < d; ++c) o[c] = exp(l1 - lse) * o1[c] + exp(l2 - lse) * o2[c];
  *l = lse;
}
