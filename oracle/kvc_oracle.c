/*
 * kvc_oracle.c -- plain CPU oracle for the decoding-time KV-cache eviction step.
 *
 * TEST INFRASTRUCTURE ONLY. Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg load this file's library. The product path never
 * calls it and shares no code, header or table with it.
 *
 * What it computes, and where each step comes from. "BeaconKV page" is the
 * article "长推理把显存吃爆了？BeaconKV：用几个「信标查询」预判模型会回头看什么"
 * (a write-up of the ICML 2026 BeaconKV paper); "ReasonAlloc page" is the note
 * "arXiv ReasonAlloc: hierarchical decoding-time KV cache" (budget source only).
 *
 *   fps        BeaconKV page, section "Continual FPS：有界内存的在线最远点采样":
 *              farthest-point sampling greedily picks m mutually most dissimilar
 *              points; the buffer is filled to B_Q^max = 32 and compressed to
 *              B_Q^min = 16. The page's formula is missing from the text; the
 *              classic greedy k-centre rule is used: start at the oldest entry,
 *              then repeatedly add the candidate whose distance to the chosen set
 *              is largest (cosine distance 1 - cos on the pre-RoPE queries;
 *              exact ties go to the lower index). Survivors keep time order.
 *   rope       BeaconKV page, section "打分时的 RoPE 对齐": beacons are rotated to
 *              the current step t, recent queries keep their own positions.
 *              Rotate-half pairing (i, i + D/2), frequency theta^(-2i/D).
 *              Rotated beacons are rounded to the cache's storage type before
 *              the dot products (the kernels multiply storage-type operands);
 *              that rounding is a quantisation decision, so the rotation that
 *              feeds it is done in binary32 like the kernels (oracle_rope_f32).
 *   score      BeaconKV page, same section: score_j = max over observation
 *              queries r of softmax_r(q_r . k_j / sqrt(D)) over all cached keys;
 *              the max also runs over the query heads sharing KV head h.
 *   variants   BeaconKV page, section "实验", the max-vs-mean ablation: the
 *              weights of one query head's observation rows may be averaged
 *              instead of maxed; the query heads of a group may be summed
 *              instead of maxed (oracle_score_agg_f64). The same function
 *              returns the head's normalised attention entropy (mean over its
 *              rows of -sum p ln p / ln N), the ReasonAlloc page's head utility
 *              signal ("Key Concepts": low entropy = focused = more budget).
 *   budget     ReasonAlloc page, "Core Mechanism": each layer's preallocated
 *              total is redistributed over its heads by utility, the total held
 *              fixed (oracle_head_budget states the rule; the page gives none).
 *   select     BeaconKV page, same section, last paragraph: prefix tokens and the
 *              most recent tokens are always kept; the rest of the budget goes
 *              to the top scores (ties: lower index). Section "实验": on reaching
 *              B_KV^max, evict 1/8 so the cache drops to 7/8 B_KV^max. ReasonAlloc
 *              page, "Core Mechanism": a per-head budget B_{L_i,H_j} caps each
 *              head instead.
 *   append     BeaconKV page, "Continual FPS" and "观察 query 集": one decode step's
 *              pre-RoPE query joins its head's buffer (compressed by FPS as soon as
 *              it is full) and its post-RoPE query joins the recent ring.
 *   epikv      EPIKV page ("方法论：EPIKV", items 1-3): a token's signal at layer l is the
 *              L2 norm of the change of the residual stream between consecutive
 *              tokens, g_l(t) = ||h_l(t) - h_l(t-1)||_2; it is made position-free by a
 *              causal rolling z-score z_l = (g_l - mu_l) / (sigma_l + eps); the
 *              eviction score is z_A - z_B for an A-band layer (kept when its signal
 *              is high) and a B-band layer (kept when low). oracle_epikv_score; the
 *              window, eps, token 0 and the std's normaliser are this build's
 *              readings (the page states none).
 *   compact    The kept tokens' K and V rows, in original order, at the head's
 *              front (out-of-place gather here); slots past the kept count keep
 *              their old contents.
 *
 * Arithmetic is fp64 throughout except the beacon rotation above; stored
 * values are rounded once, at the end, to the storage type (bf16
 * round-to-nearest-even, or fp32).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define DT_BF16 0
#define DT_F32 1

/* ------------------------------------------------------------------------- */
/* Storage conversions, from the formats' definitions.                        */
/* ------------------------------------------------------------------------- */

/* bf16 is the top half of an IEEE-754 binary32: widening is exact. */
static double bf16_bits_to_f64(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

/* Nearest bf16 to x (ties to even mantissa), computed from the value, not from
 * bit tricks: bf16 has 8 exponent bits like binary32 and 7 stored mantissa
 * bits, so its spacing at |x| in [2^E, 2^(E+1)) is 2^(E-7), with E floored at
 * -126 (subnormals). Values at or beyond the overflow midpoint become inf. */
uint16_t oracle_f64_to_bf16(double x) {
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  if (isnan(x)) return (uint16_t)(0x7fc0u | sign);
  double a = fabs(x);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(0x7f80u | sign);
  int e;
  frexp(a, &e); /* a = f * 2^e, f in [0.5, 1) -> a in [2^(e-1), 2^e) */
  int E = e - 1;
  if (E < -126) E = -126;
  double q = ldexp(1.0, E - 7);
  double n = a / q;           /* exact: scaling by a power of two */
  double r = floor(n);
  double frac = n - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  double v = r * q;           /* exact bf16 value (or 2^128 on overflow) */
  if (v >= ldexp(1.0, 128)) return (uint16_t)(0x7f80u | sign);
  float vf = (float)v;        /* exact: v has at most 8 significant bits */
  uint32_t u;
  memcpy(&u, &vf, 4);
  return (uint16_t)((u >> 16) | sign);
}

static double load_elem(const void* base, int dtype, int64_t i) {
  if (dtype == DT_BF16) return bf16_bits_to_f64(((const uint16_t*)base)[i]);
  return (double)((const float*)base)[i];
}

/* Round to the storage type and back (the value the kernels will multiply). */
static double round_to_storage(double x, int dtype) {
  if (dtype == DT_BF16) return bf16_bits_to_f64(oracle_f64_to_bf16(x));
  return (double)(float)x;
}

/* ------------------------------------------------------------------------- */
/* Farthest-point sampling (BeaconKV page, "Continual FPS").                   */
/* ------------------------------------------------------------------------- */

/* Cosine distance between rows i and j of a row-normalised matrix; a zero row
 * was left as zeros, which puts it at distance 1 from everything. */
static double cos_dist(const double* xh, int D, int i, int j) {
  double s = 0.0;
  for (int d = 0; d < D; ++d) s += xh[(int64_t)i * D + d] * xh[(int64_t)j * D + d];
  return 1.0 - s;
}

static void normalise_rows(const double* x, int n, int D, double* xh) {
  for (int i = 0; i < n; ++i) {
    double nn = 0.0;
    for (int d = 0; d < D; ++d) nn += x[(int64_t)i * D + d] * x[(int64_t)i * D + d];
    double inv = nn > 0.0 ? 1.0 / sqrt(nn) : 0.0;
    for (int d = 0; d < D; ++d) xh[(int64_t)i * D + d] = x[(int64_t)i * D + d] * inv;
  }
}

static int cmp_int(const void* a, const void* b) {
  int x = *(const int*)a, y = *(const int*)b;
  return (x > y) - (x < y);
}

/* Greedy FPS of m out of n rows of x[n][D] (fp64). Writes the picks in the
 * order they were chosen to order_out (may be NULL) and, sorted ascending, to
 * picks. gap_out (may be NULL) receives, per step k >= 1, the margin between
 * the chosen candidate's distance and the best other candidate's distance
 * (+inf when it was the only one left). Returns 0, or -1 on bad sizes. */
int oracle_fps_f64(const double* x, int n, int D, int m, int* picks, int* order_out, double* gap_out) {
  if (n < 1 || m < 1 || m > n || D < 1) return -1;
  double* xh = (double*)malloc(sizeof(double) * (size_t)n * D);
  double* mind = (double*)malloc(sizeof(double) * (size_t)n);
  char* chosen = (char*)calloc((size_t)n, 1);
  int* order = (int*)malloc(sizeof(int) * (size_t)m);
  normalise_rows(x, n, D, xh);
  order[0] = 0; /* start at the oldest buffered query */
  chosen[0] = 1;
  for (int i = 0; i < n; ++i) mind[i] = cos_dist(xh, D, i, 0);
  if (gap_out) gap_out[0] = INFINITY;
  for (int k = 1; k < m; ++k) {
    int best = -1;
    double bv = -INFINITY, second = -INFINITY;
    for (int i = 0; i < n; ++i) {
      if (chosen[i]) continue;
      if (mind[i] > bv) { second = bv; bv = mind[i]; best = i; }
      else if (mind[i] > second) second = mind[i];
    }
    order[k] = best;
    chosen[best] = 1;
    if (gap_out) gap_out[k] = bv - second;
    for (int i = 0; i < n; ++i) {
      double dd = cos_dist(xh, D, i, best);
      if (dd < mind[i]) mind[i] = dd;
    }
  }
  for (int k = 0; k < m; ++k) picks[k] = order[k];
  if (order_out) memcpy(order_out, order, sizeof(int) * (size_t)m);
  qsort(picks, (size_t)m, sizeof(int), cmp_int);
  free(xh); free(mind); free(chosen); free(order);
  return 0;
}

/* Is the ascending set `picks` (size m) a greedy FPS result of x, allowing a
 * different choice wherever the chosen candidate's distance is within tol of
 * the best one? Replays the greedy rule restricted to the set. Returns 0 if
 * valid, else 1 + the step at which no member of the set was within tol, or
 * -1 on bad input. */
int oracle_fps_check_f64(const double* x, int n, int D, const int* picks, int m, double tol) {
  if (n < 1 || m < 1 || m > n) return -1;
  for (int k = 0; k < m; ++k) {
    if (picks[k] < 0 || picks[k] >= n) return -1;
    if (k && picks[k] <= picks[k - 1]) return -1;
  }
  if (picks[0] != 0) return 1;
  double* xh = (double*)malloc(sizeof(double) * (size_t)n * D);
  double* mind = (double*)malloc(sizeof(double) * (size_t)n);
  char* chosen = (char*)calloc((size_t)n, 1);
  char* inset = (char*)calloc((size_t)n, 1);
  normalise_rows(x, n, D, xh);
  for (int k = 0; k < m; ++k) inset[picks[k]] = 1;
  chosen[0] = 1;
  for (int i = 0; i < n; ++i) mind[i] = cos_dist(xh, D, i, 0);
  int bad = 0;
  for (int k = 1; k < m && !bad; ++k) {
    double gbest = -INFINITY, sbest = -INFINITY;
    int s = -1;
    for (int i = 0; i < n; ++i) {
      if (chosen[i]) continue;
      if (mind[i] > gbest) gbest = mind[i];
      if (inset[i] && mind[i] > sbest) { sbest = mind[i]; s = i; }
    }
    if (s < 0 || sbest < gbest - tol) { bad = k + 1; break; }
    chosen[s] = 1;
    for (int i = 0; i < n; ++i) {
      double dd = cos_dist(xh, D, i, s);
      if (dd < mind[i]) mind[i] = dd;
    }
  }
  free(xh); free(mind); free(chosen); free(inset);
  return bad;
}

/* ------------------------------------------------------------------------- */
/* Rotary position encoding (BeaconKV page, "打分时的 RoPE 对齐").               */
/* ------------------------------------------------------------------------- */

void oracle_rope_f64(const double* x, int D, long long pos, double theta, double* y) {
  int h = D / 2;
  for (int i = 0; i < h; ++i) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
    double ang = (double)pos * inv_freq;
    double c = cos(ang), s = sin(ang);
    double a = x[i], b = x[i + h];
    y[i] = a * c - b * s;
    y[i + h] = b * c + a * s;
  }
}

/* The beacon rotation that feeds a rounding to the storage type. Rounding a
 * rotated beacon to bf16 is a quantisation decision, so it is taken in the
 * kernels' precision: cos/sin of the fp64 angle rounded once to binary32, then
 * each product and the difference/sum rounded to binary32 (no fused
 * multiply-add; the file is compiled with -ffp-contract=off). */
void oracle_rope_f32(const float* x, int D, long long pos, double theta, float* y) {
  int h = D / 2;
  for (int i = 0; i < h; ++i) {
    double inv_freq = pow(theta, -2.0 * (double)i / (double)D);
    double ang = (double)pos * inv_freq;
    float c = (float)cos(ang), s = (float)sin(ang);
    float a = x[i], b = x[i + h];
    float ac = a * c, bs = b * s, bc = b * c, as = a * s;
    y[i] = ac - bs;
    y[i + h] = bc + as;
  }
}

/* ------------------------------------------------------------------------- */
/* Scores (BeaconKV page, "打分时的 RoPE 对齐", the max aggregation).            */
/* ------------------------------------------------------------------------- */

/* q[M][D] observation rows, k[N][D] keys (fp64). out[j] = max_r softmax_r(j)
 * where softmax_r is over all N keys of s_rj = q_r . k_j / sqrt(D). Also
 * returns each row's log-sum-exp in lse (may be NULL). */
void oracle_score_f64(const double* q, int M, const double* k, int N, int D, double* out, double* lse) {
  double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
  double scale = 1.0 / sqrt((double)D);
  for (int j = 0; j < N; ++j) out[j] = 0.0;
  for (int r = 0; r < M; ++r) {
    double mx = -INFINITY;
    for (int j = 0; j < N; ++j) {
      double acc = 0.0;
      for (int d = 0; d < D; ++d) acc += q[(int64_t)r * D + d] * k[(int64_t)j * D + d];
      s[j] = acc * scale;
      if (s[j] > mx) mx = s[j];
    }
    double sum = 0.0;
    for (int j = 0; j < N; ++j) sum += exp(s[j] - mx);
    double l = mx + log(sum);
    if (lse) lse[r] = l;
    for (int j = 0; j < N; ++j) {
      double p = exp(s[j] - l);
      if (p > out[j]) out[j] = p;
    }
  }
  free(s);
}

/* ------------------------------------------------------------------------- */
/* Aggregation variants and attention entropy.                                 */
/* BeaconKV page, section "实验" (the max-vs-mean ablation): the softmax        */
/* weights of the observation queries may be averaged instead of maxed.        */
/* ReasonAlloc page, "Key Concepts" (Head Utility): a head's utility is its    */
/* normalised attention entropy; low entropy = focused = more useful.          */
/* ------------------------------------------------------------------------- */

#define AGG_MAX 0
#define AGG_MEAN 1
#define AGG_SUM 2

/* q[M][D] observation rows, row_head[M] the query head (0..G-1) each row
 * belongs to, k[N][D] keys (fp64). With p_rj = softmax over all N keys of
 * q_r . k_j / sqrt(D):
 *   A_g(j)  = max over the rows of head g of p_rj          (row_agg AGG_MAX)
 *           = mean over the rows of head g of p_rj         (row_agg AGG_MEAN)
 *   out[j]  = max over heads g of A_g(j)                    (group_agg AGG_MAX)
 *           = sum over heads g of A_g(j)                    (group_agg AGG_SUM)
 * Heads without rows take no part. entropy (may be NULL) receives the mean over
 * all M rows of H_r / ln N, H_r = -sum_j p_rj ln p_rj (0 when N = 1 or M = 0).
 * Returns 0, or -1 for an unknown mode or a row_head entry out of range. */
int oracle_score_agg_f64(const double* q, const int* row_head, int M, int G, const double* k, int N, int D,
                         int row_agg, int group_agg, double* out, double* entropy) {
  if ((row_agg != AGG_MAX && row_agg != AGG_MEAN) || (group_agg != AGG_MAX && group_agg != AGG_SUM)) return -1;
  for (int r = 0; r < M; ++r)
    if (row_head[r] < 0 || row_head[r] >= G) return -1;
  double* s = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
  double* A = (double*)malloc(sizeof(double) * (size_t)(N > 0 ? N : 1));
  const double scale = 1.0 / sqrt((double)D);
  double hsum = 0.0;
  for (int j = 0; j < N; ++j) out[j] = 0.0;
  for (int g = 0; g < G; ++g) {
    int Mg = 0;
    for (int j = 0; j < N; ++j) A[j] = 0.0;
    for (int r = 0; r < M; ++r) {
      if (row_head[r] != g) continue;
      ++Mg;
      double mx = -INFINITY;
      for (int j = 0; j < N; ++j) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += q[(int64_t)r * D + d] * k[(int64_t)j * D + d];
        s[j] = acc * scale;
        if (s[j] > mx) mx = s[j];
      }
      double sum = 0.0;
      for (int j = 0; j < N; ++j) sum += exp(s[j] - mx);
      const double l = mx + log(sum);
      double h = 0.0;
      for (int j = 0; j < N; ++j) {
        const double p = exp(s[j] - l);
        if (row_agg == AGG_MAX) {
          if (p > A[j]) A[j] = p;
        } else {
          A[j] += p;
        }
        if (p > 0.0) h -= p * log(p);
      }
      hsum += h;
    }
    if (Mg == 0) continue;
    for (int j = 0; j < N; ++j) {
      const double a = row_agg == AGG_MEAN ? A[j] / Mg : A[j];
      if (group_agg == AGG_SUM) out[j] += a;
      else if (a > out[j]) out[j] = a;
    }
  }
  if (entropy) *entropy = (M > 0 && N > 1) ? hsum / M / log((double)N) : 0.0;
  free(s);
  free(A);
  return 0;
}

/* Online head-wise budgets for the H KV heads of one layer of one sequence
 * (ReasonAlloc page, "Core Mechanism": budget moves from low-utility to
 * high-utility heads within a layer while the layer's preallocated total
 * stays fixed; "Key Concepts": utility from normalised attention entropy, low
 * entropy gets more). The page fixes no formula; the rule here:
 *   total  T = sum_h min(given_h, N)            (the layer's preallocation)
 *   floor  f = P + R, cap c = N - f             (every head keeps its windows)
 *   utility u_h = 1 - ent_h clipped to [0, 1], held as the integer
 *           w_h = floor(u_h * 2^24)              (24-bit fixed point)
 *   the E = T - H f slots beyond the floors are shared in proportion to w
 *   (equally when all active w are 0); a head whose share exceeds c gets c
 *   and leaves, and the rest is shared again among the others (water-filling);
 *   integer shares by largest remainder (floors, then one more slot each to the
 *   largest fractional parts, ties to the lower head index);
 *   out_h = f + share_h.
 * After w, everything is exact integer arithmetic: share_h = E_A w_h / W_A
 * with W_A = sum of the active w, compared and floored as integers. Returns 0,
 * or -1 if some given_h < P + R (the caller keeps the given budgets then). If
 * N <= f or T >= H N every head gets min(given_h, N) unchanged. H <= 64,
 * N <= 2^30. */
int oracle_head_budget(const float* ent, int H, int N, int P, int R, const int32_t* given, int32_t* out) {
  const int f = P + R;
  if (H < 1 || H > 64) return -1;
  int64_t T = 0;
  for (int h = 0; h < H; ++h) {
    if (given[h] < f) return -1;
    T += given[h] < N ? given[h] : N;
  }
  if (N <= f || T >= (int64_t)H * N) {
    for (int h = 0; h < H; ++h) out[h] = given[h] < N ? given[h] : N;
    return 0;
  }
  const int64_t cap = N - f;
  uint64_t w[64];
  int active[64];
  int64_t x[64];
  for (int h = 0; h < H; ++h) {
    double u = 1.0 - (double)ent[h];
    if (!(u > 0.0)) u = 0.0; /* also catches NaN */
    if (u > 1.0) u = 1.0;
    w[h] = (uint64_t)floor(u * 16777216.0);
    active[h] = 1;
    x[h] = 0;
  }
  /* water-filling: cap every head whose exact share E w_h / W exceeds c */
  uint64_t Erem = (uint64_t)(T - (int64_t)H * f);
  for (;;) {
    uint64_t W = 0;
    int na = 0;
    for (int h = 0; h < H; ++h)
      if (active[h]) {
        W += w[h];
        ++na;
      }
    if (na == 0) break;
    int capped = 0;
    for (int h = 0; h < H; ++h) {
      if (!active[h]) continue;
      /* share > cap  <=>  Erem w_h > cap W (or Erem > cap na for the equal split) */
      const int over = W > 0 ? Erem * w[h] > (uint64_t)cap * W : Erem > (uint64_t)cap * (uint64_t)na;
      if (over) {
        active[h] = 0;
        x[h] = cap;
        capped = 1;
      }
    }
    if (!capped) break;
    /* the capped heads take their caps out of what is shared again */
    Erem = (uint64_t)(T - (int64_t)H * f);
    for (int h = 0; h < H; ++h)
      if (!active[h]) Erem -= (uint64_t)cap;
  }
  /* floors and remainders of the active heads' exact shares */
  uint64_t W = 0;
  int na = 0;
  for (int h = 0; h < H; ++h)
    if (active[h]) {
      W += w[h];
      ++na;
    }
  uint64_t rem[64];
  uint64_t given_out = 0;
  for (int h = 0; h < H; ++h) {
    if (!active[h]) {
      rem[h] = 0;
      given_out += (uint64_t)x[h];
      continue;
    }
    const uint64_t num = W > 0 ? Erem * w[h] : Erem, den = W > 0 ? W : (uint64_t)na;
    x[h] = (int64_t)(num / den);
    rem[h] = num % den; /* remainders share the denominator: compare them directly */
    given_out += (uint64_t)x[h];
  }
  int bonus[64] = {0};
  for (uint64_t left = (uint64_t)(T - (int64_t)H * f) - given_out; left > 0; --left) {
    int best = -1;
    for (int h = 0; h < H; ++h) {
      if (!active[h] || bonus[h] || x[h] >= cap) continue;
      if (best < 0 || rem[h] > rem[best]) best = h;
    }
    if (best < 0) break; /* cannot happen: the remainders sum to fewer slots than active heads */
    bonus[best] = 1;
    x[best] += 1;
  }
  for (int h = 0; h < H; ++h) out[h] = f + (int32_t)x[h];
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Selection (BeaconKV page, end of "打分时的 RoPE 对齐"; section "实验").       */
/* ------------------------------------------------------------------------- */

static const float* g_sort_scores; /* only used inside one qsort call per thread */
#ifdef _OPENMP
#pragma omp threadprivate(g_sort_scores)
#endif

static int cmp_score_desc(const void* a, const void* b) {
  int i = *(const int*)a, j = *(const int*)b;
  float si = g_sort_scores[i], sj = g_sort_scores[j];
  if (si > sj) return -1;
  if (si < sj) return 1;
  return (i > j) - (i < j);
}

/* Keep [0,P) and [N-R,N), plus the (budget-P-R) highest-scoring middle keys
 * (ties: lower index). kept[] receives the kept indices in ascending order.
 * budget >= N keeps everything. Returns the kept count, or -1 if
 * budget < P + R (the always-kept windows would not fit). */
int oracle_select(const float* score, int N, int P, int R, int budget, int32_t* kept) {
  if (budget >= N) {
    for (int j = 0; j < N; ++j) kept[j] = j;
    return N;
  }
  if (P < 0 || R < 0 || budget < P + R) return -1;
  int mid_lo = P, mid_hi = N - R; /* middle is [P, N-R); P+R <= budget < N so it is non-empty */
  int nmid = mid_hi - mid_lo;
  int kmid = budget - P - R;
  int* idx = (int*)malloc(sizeof(int) * (size_t)(nmid > 0 ? nmid : 1));
  char* keep = (char*)calloc((size_t)N, 1);
  for (int i = 0; i < nmid; ++i) idx[i] = mid_lo + i;
  g_sort_scores = score;
  qsort(idx, (size_t)nmid, sizeof(int), cmp_score_desc);
  for (int i = 0; i < kmid; ++i) keep[idx[i]] = 1;
  for (int j = 0; j < P; ++j) keep[j] = 1;
  for (int j = mid_hi; j < N; ++j) keep[j] = 1;
  int c = 0;
  for (int j = 0; j < N; ++j)
    if (keep[j]) kept[c++] = j;
  free(idx);
  free(keep);
  return c;
}

/* ------------------------------------------------------------------------- */
/* The whole step over every (layer, batch, KV head).                          */
/* ------------------------------------------------------------------------- */

typedef struct {
  int32_t dtype; /* 0 = bf16 (uint16 bit patterns), 1 = f32 */
  int32_t L, B, Hq, Hkv, D, N;
  int32_t n_r, n_b, qmax;
  int32_t prefix, recent, budget_all;
  int64_t t;
  double theta;
  const void* K;            /* [L,B,Hkv,N,D] */
  const void* V;            /* [L,B,Hkv,N,D] */
  const void* q_recent;     /* [L,B,Hq,n_r,D], post-RoPE at their own positions */
  const void* qbuf;         /* [L,B,Hq,qmax,D], pre-RoPE, oldest first */
  const int32_t* count;     /* [L,B,Hq] */
  const int32_t* budget;    /* [L,B,Hkv] or NULL -> budget_all */
  const int32_t* forced_picks; /* [L,B,Hq,n_b] beacon rows to use instead of FPS, or NULL */
  int32_t row_agg;          /* AGG_MAX or AGG_MEAN over a query head's observation rows */
  int32_t group_agg;        /* AGG_MAX or AGG_SUM over the query heads of a KV head */
  int32_t head_budget;      /* 0: budgets as given; 1: reallocated within each layer by entropy */
  int32_t pad_;
  const float* forced_entropy; /* [L,B,Hkv] entropies for the reallocation instead of the oracle's, or NULL */
} oracle_problem;

typedef struct {
  float* scores;        /* [L,B,Hkv,N] or NULL */
  int32_t* kept_idx;    /* [L,B,Hkv,N] or NULL (entries past kept_len are -1) */
  int32_t* kept_len;    /* [L,B,Hkv] or NULL */
  void* K_out;          /* [L,B,Hkv,N,D] or NULL: a copy of K, compacted */
  void* V_out;          /* [L,B,Hkv,N,D] or NULL */
  int32_t* beacon_picks;/* [L,B,Hq,n_b] or NULL: buffer rows used as beacons (-1 = none) */
  int32_t* error;       /* [L,B,Hkv] or NULL: 0, or -1 when the head's budget was out of range */
  float* entropy;       /* [L,B,Hkv] or NULL: normalised attention entropy of the head's rows */
  int32_t* budget_used; /* [L,B,Hkv] or NULL: the budget each head was selected with */
} oracle_outputs;

/* Beacon rows of one query head: the buffer's first `count` rows if there are
 * at most n_b of them, else an FPS of n_b out of those rows (non-destructive).
 * Returns how many rows were picked. */
static int beacon_rows(const oracle_problem* p, int64_t qh, int* rows) {
  int cnt = p->count[qh];
  if (cnt < 0) cnt = 0;
  if (cnt > p->qmax) cnt = p->qmax;
  if (p->forced_picks) {
    int c = 0;
    for (int k = 0; k < p->n_b; ++k) {
      int r = p->forced_picks[qh * p->n_b + k];
      if (r >= 0) rows[c++] = r;
    }
    return c;
  }
  if (cnt <= p->n_b) {
    for (int k = 0; k < cnt; ++k) rows[k] = k;
    return cnt;
  }
  int D = p->D;
  double* x = (double*)malloc(sizeof(double) * (size_t)cnt * D);
  const int64_t base = qh * (int64_t)p->qmax * D;
  for (int i = 0; i < cnt; ++i)
    for (int d = 0; d < D; ++d) x[(int64_t)i * D + d] = load_elem(p->qbuf, p->dtype, base + (int64_t)i * D + d);
  oracle_fps_f64(x, cnt, D, p->n_b, rows, NULL, NULL);
  free(x);
  return p->n_b;
}

static void store_elem(void* base, int dtype, int64_t i, const void* src_base, int64_t si) {
  if (dtype == DT_BF16) ((uint16_t*)base)[i] = ((const uint16_t*)src_base)[si];
  else ((float*)base)[i] = ((const float*)src_base)[si];
}

/* Scores (and the entropy) of one KV head. */
static void score_head(const oracle_problem* p, const oracle_outputs* o, int64_t head, float* scf, double* ent) {
  const int D = p->D, N = p->N, G = p->Hq / p->Hkv;
  const int l = (int)(head / ((int64_t)p->B * p->Hkv));
  const int b = (int)((head / p->Hkv) % p->B);
  const int h = (int)(head % p->Hkv);
  const int maxrows = G * (p->n_r + p->n_b);
  double* q = (double*)malloc(sizeof(double) * (size_t)(maxrows > 0 ? maxrows : 1) * D);
  int* row_head = (int*)malloc(sizeof(int) * (size_t)(maxrows > 0 ? maxrows : 1));
  double* k = (double*)malloc(sizeof(double) * (size_t)N * D);
  double* sc = (double*)malloc(sizeof(double) * (size_t)N);
  int* rows = (int*)malloc(sizeof(int) * (size_t)(p->qmax > 0 ? p->qmax : 1));
  float* tmp = (float*)malloc(sizeof(float) * (size_t)D);
  float* rot = (float*)malloc(sizeof(float) * (size_t)D);

  /* observation rows: for each query head of the group, its recent queries as
   * stored, then its beacons rotated to step t and rounded to storage type */
  int M = 0;
  for (int g = 0; g < G; ++g) {
    const int hq = h * G + g;
    const int64_t qh = ((int64_t)l * p->B + b) * p->Hq + hq;
    for (int r = 0; r < p->n_r; ++r, ++M) {
      row_head[M] = g;
      for (int d = 0; d < D; ++d)
        q[(int64_t)M * D + d] = load_elem(p->q_recent, p->dtype, (qh * p->n_r + r) * D + d);
    }
    int nb = beacon_rows(p, qh, rows);
    if (o->beacon_picks)
      for (int kk = 0; kk < p->n_b; ++kk) o->beacon_picks[qh * p->n_b + kk] = kk < nb ? rows[kk] : -1;
    for (int kk = 0; kk < nb; ++kk, ++M) {
      row_head[M] = g;
      for (int d = 0; d < D; ++d) tmp[d] = (float)load_elem(p->qbuf, p->dtype, (qh * p->qmax + rows[kk]) * D + d);
      oracle_rope_f32(tmp, D, (long long)p->t, p->theta, rot);
      for (int d = 0; d < D; ++d) q[(int64_t)M * D + d] = round_to_storage((double)rot[d], p->dtype);
    }
  }
  const int64_t kbase = head * (int64_t)N * D;
  for (int64_t i = 0; i < (int64_t)N * D; ++i) k[i] = load_elem(p->K, p->dtype, kbase + i);
  if (p->row_agg == AGG_MAX && p->group_agg == AGG_MAX && !o->entropy && !p->head_budget) {
    oracle_score_f64(q, M, k, N, D, sc, NULL);
    *ent = 0.0;
  } else {
    oracle_score_agg_f64(q, row_head, M, G, k, N, D, p->row_agg, p->group_agg, sc, ent);
  }
  for (int j = 0; j < N; ++j) scf[j] = (float)sc[j];
  if (o->scores) memcpy(&o->scores[head * N], scf, sizeof(float) * (size_t)N);
  if (o->entropy) o->entropy[head] = (float)*ent;
  free(q); free(row_head); free(k); free(sc); free(rows); free(tmp); free(rot);
}

/* Selection and compaction of one KV head with the given budget. */
static void keep_head(const oracle_problem* p, const oracle_outputs* o, int64_t head, const float* scf, int budget) {
  const int D = p->D, N = p->N;
  int32_t* kept = (int32_t*)malloc(sizeof(int32_t) * (size_t)N);
  if (o->budget_used) o->budget_used[head] = budget;
  int len = oracle_select(scf, N, p->prefix, p->recent, budget, kept);
  if (o->error) o->error[head] = len < 0 ? -1 : 0;
  if (len < 0) { /* out-of-range budget: the head is left whole */
    for (int j = 0; j < N; ++j) kept[j] = j;
    len = N;
  }
  if (o->kept_len) o->kept_len[head] = len;
  if (o->kept_idx)
    for (int j = 0; j < N; ++j) o->kept_idx[head * N + j] = j < len ? kept[j] : -1;
  /* compaction: out-of-place gather into the output copies */
  const int64_t kbase = head * (int64_t)N * D;
  if (o->K_out)
    for (int j = 0; j < len; ++j)
      for (int d = 0; d < D; ++d) store_elem(o->K_out, p->dtype, kbase + (int64_t)j * D + d, p->K, kbase + (int64_t)kept[j] * D + d);
  if (o->V_out)
    for (int j = 0; j < len; ++j)
      for (int d = 0; d < D; ++d) store_elem(o->V_out, p->dtype, kbase + (int64_t)j * D + d, p->V, kbase + (int64_t)kept[j] * D + d);
  free(kept);
}

/* The eviction step for every (l, b, h_kv), in three steps: the scores (and
 * entropy) of each head; with head_budget = 1 the budgets of each layer of each
 * sequence (oracle_head_budget over its Hkv heads); then selection and
 * compaction of each head. K_out / V_out must already hold a copy of K / V
 * (slots past the kept count are left as they are). heads / nheads (optional)
 * restrict the work to the listed flat head ids (l*B + b)*Hkv + h; with
 * head_budget = 1 the other heads of each listed head's layer are scored too,
 * since its budget depends on them. Returns 0, or -1 on bad sizes or modes. */
int oracle_evict(const oracle_problem* p, const oracle_outputs* o, const int64_t* heads, int64_t nheads) {
  if (!p || !o || p->L < 1 || p->B < 1 || p->Hkv < 1 || p->Hq < p->Hkv || p->Hq % p->Hkv) return -1;
  if (p->D < 2 || p->D % 2 || p->N < 1 || p->n_r < 0 || p->n_b < 0 || p->qmax < 0) return -1;
  if ((p->row_agg != AGG_MAX && p->row_agg != AGG_MEAN) || (p->group_agg != AGG_MAX && p->group_agg != AGG_SUM) ||
      p->head_budget < 0 || p->head_budget > 1 || p->Hkv > 64)
    return -1;
  const int64_t total = (int64_t)p->L * p->B * p->Hkv;
  const int N = p->N, Hkv = p->Hkv;
  /* which heads to score (want = 1) and to keep (want = 2) */
  char* want = (char*)calloc((size_t)total, 1);
  for (int64_t i = 0; i < (heads ? nheads : total); ++i) {
    const int64_t head = heads ? heads[i] : i;
    if (head < 0 || head >= total) continue;
    want[head] = 2;
    if (p->head_budget)
      for (int64_t g = head - head % Hkv; g < head - head % Hkv + Hkv; ++g)
        if (!want[g]) want[g] = 1;
  }
  float* scf = (float*)malloc(sizeof(float) * (size_t)total * N);
  double* ent = (double*)calloc((size_t)total, sizeof(double));
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t head = 0; head < total; ++head)
    if (want[head]) score_head(p, o, head, scf + head * N, &ent[head]);
  int32_t* bud = (int32_t*)malloc(sizeof(int32_t) * (size_t)total);
  for (int64_t head = 0; head < total; ++head) bud[head] = p->budget ? p->budget[head] : p->budget_all;
  if (p->head_budget)
    for (int64_t lb = 0; lb < total / Hkv; ++lb) {
      if (!want[lb * Hkv]) continue;
      float e[64];
      int32_t out[64];
      for (int h = 0; h < Hkv; ++h)
        e[h] = p->forced_entropy ? p->forced_entropy[lb * Hkv + h] : (float)ent[lb * Hkv + h];
      if (oracle_head_budget(e, Hkv, N, p->prefix, p->recent, bud + lb * Hkv, out) == 0)
        memcpy(bud + lb * Hkv, out, sizeof(int32_t) * (size_t)Hkv);
    }
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t head = 0; head < total; ++head)
    if (want[head] == 2) keep_head(p, o, head, scf + head * N, bud[head]);
  free(want); free(scf); free(ent); free(bud);
  return 0;
}

/* Continual-FPS compression of every query head whose buffer is full: the
 * qmax buffered pre-RoPE queries are cut to qmax/2 by FPS, the survivors move
 * to the buffer's front in time order and count becomes qmax/2. Heads with
 * count < qmax are left alone. picks [L*B*Hq, qmax/2] (may be NULL) receives
 * the surviving rows' old indices (-1 for heads left alone). Returns the
 * number of compressed heads, or -1 on bad sizes. */
int oracle_fps_update(int32_t dtype, int32_t nheads_q, int32_t D, void* qbuf, int32_t qmax, int32_t* count,
                      int32_t* picks) {
  if (nheads_q < 0 || D < 1 || qmax < 2 || qmax % 2) return -1;
  const int m = qmax / 2;
  int done = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : done)
  for (int64_t qh = 0; qh < nheads_q; ++qh) {
    if (count[qh] != qmax) {
      if (picks)
        for (int k = 0; k < m; ++k) picks[qh * m + k] = -1;
      continue;
    }
    double* x = (double*)malloc(sizeof(double) * (size_t)qmax * D);
    int* sel = (int*)malloc(sizeof(int) * (size_t)m);
    const int64_t base = qh * (int64_t)qmax * D;
    for (int i = 0; i < qmax; ++i)
      for (int d = 0; d < D; ++d) x[(int64_t)i * D + d] = load_elem(qbuf, dtype, base + (int64_t)i * D + d);
    oracle_fps_f64(x, qmax, D, m, sel, NULL, NULL);
    /* sel is ascending and sel[k] >= k, so a forward copy never overwrites a
     * row that is still to be read */
    for (int k = 0; k < m; ++k)
      for (int d = 0; d < D; ++d) store_elem(qbuf, dtype, base + (int64_t)k * D + d, qbuf, base + (int64_t)sel[k] * D + d);
    count[qh] = m;
    if (picks)
      for (int k = 0; k < m; ++k) picks[qh * m + k] = sel[k];
    free(x);
    free(sel);
    done += 1;
  }
  return done;
}

/* Compress one full buffer (qmax rows at base) to qmax/2 survivors in time order;
 * sel receives the survivors' old rows. */
static void compress_one(int32_t dtype, int32_t D, void* qbuf, int64_t base, int32_t qmax, int* sel) {
  const int m = qmax / 2;
  double* x = (double*)malloc(sizeof(double) * (size_t)qmax * D);
  for (int i = 0; i < qmax; ++i)
    for (int d = 0; d < D; ++d) x[(int64_t)i * D + d] = load_elem(qbuf, dtype, base + (int64_t)i * D + d);
  oracle_fps_f64(x, qmax, D, m, sel, NULL, NULL);
  for (int k = 0; k < m; ++k)
    for (int d = 0; d < D; ++d) store_elem(qbuf, dtype, base + (int64_t)k * D + d, qbuf, base + (int64_t)sel[k] * D + d);
  free(x);
}

/* One decode step's queries into the observation state (BeaconKV page, "Continual FPS": the
 * buffer of pre-RoPE queries grows to B_Q^max and is then cut back to B_Q^min; "观察 query 集":
 * the recent queries are the latest n_r at their own positions). For every query head:
 *   - a buffer already full on entry (count == qmax) is compressed first;
 *   - the new pre-RoPE query q_pre goes to buffer row count, count += 1;
 *   - a buffer that has just become full is compressed (FPS to qmax/2, time order);
 *   - ring row t mod n_r of q_recent receives q_post, or when q_post is NULL the binary32
 *     rotation of q_pre to position t rounded to the storage type (as for beacons).
 * A count outside [0, qmax] leaves that head's buffer alone (error[qh] = -1); its ring row is
 * still written. picks [nheads_q, qmax/2] (may be NULL) receives the old rows of the last
 * compression in this call, -1 when none. Returns the number of compressions, or -1 on bad
 * sizes. */
int oracle_append(int32_t dtype, int32_t nheads_q, int32_t D, const void* q_pre, const void* q_post, int64_t t,
                  double theta, void* qbuf, int32_t qmax, int32_t* count, void* q_recent, int32_t n_r,
                  int32_t* picks, int32_t* error) {
  if (nheads_q < 0 || D < 2 || D % 2 || qmax < 2 || qmax % 2 || n_r < 0 || t < 0) return -1;
  const int m = qmax / 2;
  int done = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : done)
  for (int64_t qh = 0; qh < nheads_q; ++qh) {
    int* sel = (int*)malloc(sizeof(int) * (size_t)m);
    float* tmp = (float*)malloc(sizeof(float) * (size_t)D);
    float* rot = (float*)malloc(sizeof(float) * (size_t)D);
    int compressed = 0;
    if (error) error[qh] = 0;
    if (n_r > 0) {
      const int64_t dst = (qh * n_r + t % n_r) * (int64_t)D;
      if (q_post) {
        for (int d = 0; d < D; ++d) store_elem(q_recent, dtype, dst + d, q_post, qh * (int64_t)D + d);
      } else {
        for (int d = 0; d < D; ++d) tmp[d] = (float)load_elem(q_pre, dtype, qh * (int64_t)D + d);
        oracle_rope_f32(tmp, D, (long long)t, theta, rot);
        for (int d = 0; d < D; ++d) {
          const double v = round_to_storage((double)rot[d], dtype);
          if (dtype == DT_BF16) ((uint16_t*)q_recent)[dst + d] = oracle_f64_to_bf16(v);
          else ((float*)q_recent)[dst + d] = (float)v;
        }
      }
    }
    int c = count[qh];
    const int64_t base = qh * (int64_t)qmax * D;
    if (c < 0 || c > qmax) {
      if (error) error[qh] = -1;
    } else {
      if (c == qmax) {
        compress_one(dtype, D, qbuf, base, qmax, sel);
        c = m;
        compressed = 1;
      }
      for (int d = 0; d < D; ++d) store_elem(qbuf, dtype, base + (int64_t)c * D + d, q_pre, qh * (int64_t)D + d);
      c += 1;
      if (c == qmax) {
        compress_one(dtype, D, qbuf, base, qmax, sel);
        c = m;
        compressed += 1;
      }
      count[qh] = c;
    }
    if (picks)
      for (int k = 0; k < m; ++k) picks[qh * m + k] = compressed ? sel[k] : -1;
    done += compressed;
    free(sel);
    free(tmp);
    free(rot);
  }
  return done;
}

/* The z-score half of oracle_epikv_score, from given signals g [2][B][N] (layer A, layer B). */
int oracle_epikv_z(int32_t B, int32_t N, const double* g, int32_t W, double eps, double* score) {
  if (B < 0 || N < 0 || W < 1 || !(eps >= 0.0)) return -1;
#pragma omp parallel for schedule(static)
  for (int64_t bt = 0; bt < (int64_t)B * N; ++bt) {
    const int64_t b = bt / N, t = bt % N;
    double z[2] = {0.0, 0.0};
    if (t >= 1) {
      const int64_t lo = t - W + 1 > 1 ? t - W + 1 : 1;
      const double n = (double)(t - lo + 1);
      for (int layer = 0; layer < 2; ++layer) {
        const double* gl = g + ((int64_t)layer * B + b) * N;
        double sum = 0.0;
        for (int64_t u = lo; u <= t; ++u) sum += gl[u];
        const double mu = sum / n;
        double var = 0.0;
        for (int64_t u = lo; u <= t; ++u) var += (gl[u] - mu) * (gl[u] - mu);
        const double sigma = sqrt(var / n);
        z[layer] = (gl[t] - mu) / (sigma + eps);
      }
    }
    score[b * N + t] = z[0] - z[1];
  }
  return 0;
}

/* EPIKV page, "方法论：EPIKV": the epiphany signal and its causal rolling z-score, per
 * sequence b of B, for the hidden states of two layers hA, hB [B][N][dm] (storage
 * type dtype). Readings (the page gives no window, eps or first-token rule):
 *   g(0) = 0 (token 0 has no predecessor) and token 0 lies in no window;
 *   for t >= 1: g(t) = sqrt(sum_i (h(t)_i - h(t-1)_i)^2);
 *   window(t) = tokens max(1, t - W + 1) .. t (causal, t itself included), n = min(t, W);
 *   mu(t) = mean of g over window(t); sigma(t) = sqrt(mean of (g - mu)^2) (population);
 *   z(t) = (g(t) - mu(t)) / (sigma(t) + eps) for t >= 1, z(0) = 0;
 *   score(t) = zA(t) - zB(t).
 * Outputs (fp64): g [2][B][N] (may be NULL) and score [B][N]. Returns 0, or -1 on bad sizes. */
int oracle_epikv_score(int32_t dtype, int32_t B, int32_t N, int32_t dm, const void* hA, const void* hB, int32_t W,
                       double eps, double* g_out, double* score) {
  if (B < 0 || N < 0 || dm < 1 || W < 1 || !(eps >= 0.0)) return -1;
  double* g = (double*)malloc(sizeof(double) * 2 * (size_t)(B > 0 ? B : 1) * (size_t)(N > 0 ? N : 1));
#pragma omp parallel for schedule(static)
  for (int64_t bt = 0; bt < (int64_t)B * N; ++bt) {
    const int64_t b = bt / N, t = bt % N;
    for (int layer = 0; layer < 2; ++layer) {
      const void* h = layer == 0 ? hA : hB;
      double ss = 0.0;
      if (t >= 1)
        for (int i = 0; i < dm; ++i) {
          const double d = load_elem(h, dtype, (b * N + t) * dm + i) - load_elem(h, dtype, (b * N + t - 1) * dm + i);
          ss += d * d;
        }
      g[((int64_t)layer * B + b) * N + t] = sqrt(ss);
    }
  }
  oracle_epikv_z(B, N, g, W, eps, score);
  if (g_out) memcpy(g_out, g, sizeof(double) * 2 * (size_t)B * (size_t)N);
  free(g);
  return 0;
}

int oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
  return omp_get_max_threads();
#else
  (void)n;
  return 1;
#endif
}
