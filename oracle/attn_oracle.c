/*
 * attn_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of exact attention with explicit masks.
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg may load
 * this code; the product path never calls it and shares no code with it.
 *
 * What it computes, row by row (no tiling, no fusion, no online softmax):
 *
 *   s_ij  = scale * sum_t q_it k_jt                for j in A(i)
 *   M_i   = max_{j in A(i)} s_ij
 *   l_i   = sum_{j in A(i)} exp(s_ij - M_i)
 *   o_i   = sum_{j in A(i)} exp(s_ij - M_i) v_j / l_i
 *   lse_i = M_i + ln l_i
 *
 * Sources:
 *   - "Fused Self Attention" (NKI tutorial), section "Background": S = Q K^T,
 *     R = softmax(S) V over (seqlen, d_head) operands.
 *   - "Profiling in PyTorch" part 3, section "Deconstructing Naive Attention":
 *     scores are multiplied by scale = 1/sqrt(head_dim), masked positions are
 *     filled with -inf, a row softmax follows, then the product with v.
 *   - NATTEN issue #142 ("circular windowed attention"): a query attends the
 *     keys between its window start and window end; in wrap mode the window
 *     wraps around the borders like a circularly padded convolution, and the
 *     worked example (5x5 grid, kernel 3) gives every query exactly 9 keys.
 *     The forward returns a float32 logsumexp of shape q.shape[:-1]; here it
 *     is the natural log of sum_{j in A(i)} exp(s_ij).
 *
 * Allowed sets A(i) (mask_kind):
 *   0 NONE   : every key j < Nk.
 *   1 CAUSAL : j <= i (top-left alignment, as is_causal=True).
 *   4 CAUSAL_BR : j <= i + (Nk - Nq) (bottom-right alignment: the last query
 *              sees every key, as when the queries are the newest Nq of Nk
 *              tokens). With Nq > Nk the first Nq - Nk rows see no key.
 *   2 NA2D   : tokens are laid out row-major on a grid_h x grid_w grid;
 *              query (qy, qx), key (ky, kx); the key is allowed iff both axes
 *              are allowed by the one-axis rule below, each axis with its own
 *              window size (odd) and its own choice of clamp or wrap; one
 *              dilation for both. A grid with one row and a window of 1 along
 *              it is 1-D neighbourhood attention.
 *     clamp: the window keeps its full size k and is shifted inward at the
 *              borders. With dilation delta, keys share the query's residue
 *              modulo delta, and the dilation-1 rule is applied to the index
 *              inside that residue class.
 *     wrap : the keys are (q + delta*t) mod G for t in [-k/2, k/2].
 *   3 NA3D   : tokens are laid out row-major on a grid_d x grid_h x grid_w
 *              volume (depth slowest); query (qt, qy, qx), key (kt, ky, kx);
 *              the key is allowed iff all three axes are allowed by the same
 *              one-axis rule, each axis with its own window and its own clamp
 *              or wrap choice; one dilation for all three. The NATTEN issue's
 *              requester works with 3-D volumes (about 15-20 patches a side,
 *              window 5) and wraps some of the axes.
 *   A row whose allowed set is empty gets o = 0 and lse = -inf (the
 *   NaN-guarding convention of a "safe" softmax).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MASK_NONE 0
#define ORACLE_MASK_CAUSAL 1
#define ORACLE_MASK_NA2D 2
#define ORACLE_MASK_NA3D 3
#define ORACLE_MASK_CAUSAL_BR 4

typedef struct {
  int Nq, Nk, d;
  double scale;
  int mask_kind, window_h, window_w, dilation, wrap_h, wrap_w, grid_h, grid_w;
  int window_d, wrap_d, grid_d; /* NA3D's depth axis */
} problem_t;

/* One axis of the clamped neighbourhood: is key coordinate kc in the window of
 * query coordinate qc on an axis of length G?  Window size k (odd), dilation dl. */
static int axis_allowed_clamp(int qc, int kc, int G, int k, int dl) {
  int residue = qc % dl;
  if (kc % dl != residue) return 0;
  /* number of grid positions that share this residue */
  int len = (G - residue + dl - 1) / dl;
  int a = qc / dl;     /* query index inside its residue class */
  int b = kc / dl;     /* key index inside the same class       */
  int start = a - k / 2;
  if (start < 0) start = 0;
  if (start > len - k) start = len - k;
  return b >= start && b < start + k;
}

/* One axis of the circular ("wrap") neighbourhood. */
static int axis_allowed_wrap(int qc, int kc, int G, int k, int dl) {
  int half = k / 2;
  for (int t = -half; t <= half; ++t) {
    int c = qc + dl * t;
    c %= G;
    if (c < 0) c += G;
    if (c == kc) return 1;
  }
  return 0;
}

static int axis_allowed(int wrap, int qc, int kc, int G, int k, int dl) {
  return wrap ? axis_allowed_wrap(qc, kc, G, k, dl) : axis_allowed_clamp(qc, kc, G, k, dl);
}

static int allowed(const problem_t* p, int i, int j) {
  switch (p->mask_kind) {
    case ORACLE_MASK_NONE:
      return 1;
    case ORACLE_MASK_CAUSAL:
      return j <= i;
    case ORACLE_MASK_CAUSAL_BR:
      return (int64_t)j <= (int64_t)i + (p->Nk - p->Nq);
    case ORACLE_MASK_NA2D: {
      int qy = i / p->grid_w, qx = i % p->grid_w;
      int ky = j / p->grid_w, kx = j % p->grid_w;
      const int row_ok = p->wrap_h ? axis_allowed_wrap(qy, ky, p->grid_h, p->window_h, p->dilation)
                                   : axis_allowed_clamp(qy, ky, p->grid_h, p->window_h, p->dilation);
      const int col_ok = p->wrap_w ? axis_allowed_wrap(qx, kx, p->grid_w, p->window_w, p->dilation)
                                   : axis_allowed_clamp(qx, kx, p->grid_w, p->window_w, p->dilation);
      return row_ok && col_ok;
    }
    case ORACLE_MASK_NA3D: {
      const int plane = p->grid_h * p->grid_w;
      int qt = i / plane, qy = (i % plane) / p->grid_w, qx = i % p->grid_w;
      int kt = j / plane, ky = (j % plane) / p->grid_w, kx = j % p->grid_w;
      return axis_allowed(p->wrap_d, qt, kt, p->grid_d, p->window_d, p->dilation) &&
             axis_allowed(p->wrap_h, qy, ky, p->grid_h, p->window_h, p->dilation) &&
             axis_allowed(p->wrap_w, qx, kx, p->grid_w, p->window_w, p->dilation);
    }
    default:
      return 0;
  }
}

/* Returns 0 on success, -1 on bad arguments, -2 on allocation failure. */
static int check_args(const problem_t* p, int B, int H) {
  if (B < 1 || H < 1 || p->Nq < 1 || p->Nk < 1 || p->d < 1) return -1;
  if (p->mask_kind < 0 || p->mask_kind > 4) return -1;
  if (p->mask_kind == ORACLE_MASK_NA3D) {
    if (p->grid_d < 1 || p->window_d < 1 || p->window_d % 2 == 0) return -1;
    if (p->window_d > 1 && (int64_t)p->window_d * p->dilation > p->grid_d) return -1;
  }
  if (p->mask_kind == ORACLE_MASK_NA2D || p->mask_kind == ORACLE_MASK_NA3D) {
    const int64_t depth = p->mask_kind == ORACLE_MASK_NA3D ? p->grid_d : 1;
    if (p->grid_h < 1 || p->grid_w < 1) return -1;
    if (depth * p->grid_h * p->grid_w != p->Nq || p->Nq != p->Nk) return -1;
    if (p->window_h < 1 || p->window_h % 2 == 0 || p->window_w < 1 || p->window_w % 2 == 0)
      return -1;
    if (p->dilation < 1) return -1;
    /* every residue class of an axis holds at least k members (clamp), and the
     * k wrapped keys are distinct (wrap), iff k = 1 or k * dilation <= G */
    if (p->window_h > 1 && p->window_h * p->dilation > p->grid_h) return -1;
    if (p->window_w > 1 && p->window_w * p->dilation > p->grid_w) return -1;
  }
  return 0;
}

/* One output row: flat row index r in [0, B*H*Nq).  scores: scratch of Nk. */
static void one_row(const problem_t* p, const double* q, const double* k,
                    const double* v, int64_t r, double* o_row, double* lse_out,
                    double* scores, unsigned char* ok) {
  const int Nq = p->Nq, Nk = p->Nk, d = p->d;
  const int64_t bh = r / Nq;
  const int i = (int)(r % Nq);
  const double* qi = q + r * d;
  const double* kb = k + bh * (int64_t)Nk * d;
  const double* vb = v + bh * (int64_t)Nk * d;

  double M = -INFINITY;
  int any = 0;
  for (int j = 0; j < Nk; ++j) {
    ok[j] = (unsigned char)allowed(p, i, j);
    if (!ok[j]) continue;
    const double* kj = kb + (int64_t)j * d;
    double dot = 0.0;
    for (int t = 0; t < d; ++t) dot += qi[t] * kj[t];
    scores[j] = p->scale * dot;
    if (!any || scores[j] > M) M = scores[j];
    any = 1;
  }
  for (int t = 0; t < d; ++t) o_row[t] = 0.0;
  if (!any) {
    *lse_out = -INFINITY;
    return;
  }
  double l = 0.0;
  for (int j = 0; j < Nk; ++j) {
    if (!ok[j]) continue;
    double w = exp(scores[j] - M);
    l += w;
    const double* vj = vb + (int64_t)j * d;
    for (int t = 0; t < d; ++t) o_row[t] += w * vj[t];
  }
  for (int t = 0; t < d; ++t) o_row[t] /= l;
  *lse_out = M + log(l);
}

/*
 * q: [B,H,Nq,d], k,v: [B,H,Nk,d], all fp64 contiguous.
 * rows == NULL: every row; o is [B,H,Nq,d], lse is [B,H,Nq].
 * rows != NULL: nrows flat row indices in [0, B*H*Nq); o is [nrows,d], lse [nrows].
 * window_h / window_w and wrap_h / wrap_w: the row (grid_h) and column (grid_w)
 * axes of NA2D and NA3D; window_d / wrap_d / grid_d: NA3D's depth axis; all
 * ignored for the other masks.
 * nthreads <= 0 leaves the OpenMP default.
 */
int oracle_attn_rows(const double* q, const double* k, const double* v,
                     double* o, double* lse, int B, int H, int Nq, int Nk, int d,
                     double scale, int mask_kind, int window_h, int window_w, int dilation,
                     int wrap_h, int wrap_w, int grid_h, int grid_w, int window_d, int wrap_d,
                     int grid_d, const int64_t* rows, int64_t nrows, int nthreads) {
  problem_t p = {Nq, Nk, d, scale, mask_kind, window_h, window_w, dilation,
                 wrap_h, wrap_w, grid_h, grid_w, window_d, wrap_d, grid_d};
  if (check_args(&p, B, H) != 0) return -1;
  const int64_t total = (int64_t)B * H * Nq;
  const int64_t n = rows ? nrows : total;
  if (rows) {
    for (int64_t x = 0; x < n; ++x)
      if (rows[x] < 0 || rows[x] >= total) return -1;
  }
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int failed = 0;
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)Nk);
    unsigned char* ok = (unsigned char*)malloc((size_t)Nk);
    if (!scores || !ok) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (int64_t x = 0; x < n; ++x) {
        int64_t r = rows ? rows[x] : x;
        one_row(&p, q, k, v, r, o + x * d, lse + x, scores, ok);
      }
    }
    free(scores);
    free(ok);
  }
  return failed ? -2 : 0;
}

/*
 * Backward pass (the gradients of a scalar loss L through the forward above),
 * for one (batch, head), row by row in fp64. With P_ij = exp(s_ij - lse_i) the
 * softmax weights of row i (0 outside A(i)) and dO the gradient of L at O:
 *   dV_j  = sum_i P_ij dO_i
 *   dP_ij = dO_i . v_j
 *   D_i   = dO_i . o_i              (= sum_j P_ij dP_ij)
 *   dS_ij = P_ij (dP_ij - D_i)       (the softmax Jacobian applied to dP)
 *   dQ_i  = scale sum_j dS_ij k_j,   dK_j = scale sum_i dS_ij q_i
 * which is the chain rule through s = scale q.k, the row softmax and o = P v.
 * Sources: the forward's sources above (S = Q K^T, the row softmax, R = S V);
 * the backward itself is the textbook chain rule.
 */
static void one_head_bwd(const problem_t* p, const double* q, const double* k, const double* v,
                         const double* dout, double* dq, double* dk, double* dv, double* s,
                         unsigned char* ok, double* pw, double* dp) {
  const int Nq = p->Nq, Nk = p->Nk, d = p->d;
  for (int64_t x = 0; x < (int64_t)Nk * d; ++x) { dk[x] = 0.0; dv[x] = 0.0; }
  for (int i = 0; i < Nq; ++i) {
    const double* qi = q + (int64_t)i * d;
    const double* gi = dout + (int64_t)i * d;
    double M = -INFINITY;
    int any = 0;
    for (int j = 0; j < Nk; ++j) {
      ok[j] = (unsigned char)allowed(p, i, j);
      if (!ok[j]) continue;
      double dot = 0.0;
      for (int t = 0; t < d; ++t) dot += qi[t] * k[(int64_t)j * d + t];
      s[j] = p->scale * dot;
      if (!any || s[j] > M) M = s[j];
      any = 1;
    }
    double* dqi = dq + (int64_t)i * d;
    for (int t = 0; t < d; ++t) dqi[t] = 0.0;
    if (!any) continue;
    double l = 0.0;
    for (int j = 0; j < Nk; ++j)
      if (ok[j]) l += exp(s[j] - M);
    /* o_i (for D_i), the weights P_ij and dP_ij */
    double Di = 0.0;
    for (int t = 0; t < d; ++t) {
      double ot = 0.0;
      for (int j = 0; j < Nk; ++j)
        if (ok[j]) ot += exp(s[j] - M) / l * v[(int64_t)j * d + t];
      Di += gi[t] * ot;
    }
    for (int j = 0; j < Nk; ++j) {
      if (!ok[j]) continue;
      pw[j] = exp(s[j] - M) / l;
      double g = 0.0;
      for (int t = 0; t < d; ++t) g += gi[t] * v[(int64_t)j * d + t];
      dp[j] = g;
    }
    for (int j = 0; j < Nk; ++j) {
      if (!ok[j]) continue;
      const double dsij = pw[j] * (dp[j] - Di);
      for (int t = 0; t < d; ++t) {
        dqi[t] += p->scale * dsij * k[(int64_t)j * d + t];
        dk[(int64_t)j * d + t] += p->scale * dsij * qi[t];
        dv[(int64_t)j * d + t] += pw[j] * gi[t];
      }
    }
  }
}

/*
 * q, dout: [B,H,Nq,d]; k, v: [B,H,Nk,d]; outputs dq [B,H,Nq,d], dk and dv
 * [B,H,Nk,d]; all fp64 contiguous. Mask arguments as oracle_attn_rows.
 */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv, int B, int H, int Nq, int Nk, int d,
                    double scale, int mask_kind, int window_h, int window_w, int dilation,
                    int wrap_h, int wrap_w, int grid_h, int grid_w, int window_d, int wrap_d,
                    int grid_d, int nthreads) {
  problem_t p = {Nq, Nk, d, scale, mask_kind, window_h, window_w, dilation,
                 wrap_h, wrap_w, grid_h, grid_w, window_d, wrap_d, grid_d};
  if (check_args(&p, B, H) != 0) return -1;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int failed = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)Nk * 3);
    unsigned char* ok = (unsigned char*)malloc((size_t)Nk);
    if (!s || !ok) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (int64_t bh = 0; bh < (int64_t)B * H; ++bh) {
        const int64_t qo = bh * (int64_t)Nq * d, ko = bh * (int64_t)Nk * d;
        one_head_bwd(&p, q + qo, k + ko, v + ko, dout + qo, dq + qo, dk + ko, dv + ko, s, ok,
                     s + Nk, s + 2 * (int64_t)Nk);
      }
    }
    free(s);
    free(ok);
  }
  return failed ? -2 : 0;
}

/* Number of threads the OpenMP runtime will use (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* The allowed-set predicate itself, exposed so tests can inspect masks. */
int oracle_allowed(int i, int j, int Nq, int Nk, int mask_kind, int window_h, int window_w,
                   int dilation, int wrap_h, int wrap_w, int grid_h, int grid_w, int window_d,
                   int wrap_d, int grid_d) {
  problem_t p = {Nq, Nk, 1, 1.0, mask_kind, window_h, window_w, dilation,
                 wrap_h, wrap_w, grid_h, grid_w, window_d, wrap_d, grid_d};
  if (check_args(&p, 1, 1) != 0) return -1;
  if (i < 0 || i >= Nq || j < 0 || j >= Nk) return -1;
  return allowed(&p, i, j);
}
