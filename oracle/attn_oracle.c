/*
 * Plain fp64 CPU oracle for causal grouped-query attention with rotary
 * position embedding on Q and K (forward and backward).
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link or call this
 * file: only the test-suite, the smoke check and the CPU-baseline leg of the
 * benchmark use it. It shares no code, header, table or constant with the CUDA
 * library; the two meet only in the seeded inputs they are both given.
 *
 * What it computes follows the NanoEuler pages:
 *   - "Architecture": decoder-only transformer, rotary position embedding
 *     applied to queries and keys, grouped-query attention in which query
 *     heads share a smaller set of key/value heads (mynewscn README;
 *     socker-news README, "Architecture" / "Basic configuration").
 *   - "GPU engine": hand-written FlashAttention that is tiled, uses an online
 *     softmax and never forms the T x T matrix (socker-news README,
 *     "Kernels and acceleration"; ojeo summary). FlashAttention reaches the
 *     same result as plain causal softmax attention, so this oracle is that
 *     plain definition written out, one query row (or one key row) at a time.
 *   - causal mask: keys after the query are excluded (openai-hub article,
 *     section on the softmax kernel's causal mask).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - RoPE pairs are interleaved (x[2i], x[2i+1]), angle t * theta_i with
 *     theta_i = base^(-2i/D), rotation [[cos, -sin], [sin, cos]], positions
 *     t = 0..T-1 for both queries and keys.  The pages name no pair layout;
 *     `half` selects the other common reading, pairs (x[i], x[i + D/2]) with
 *     the same angles (the half-split layout).
 *   - softmax scale is 1/sqrt(D), applied to the dot product of the rotated
 *     vectors; key j is visible to query t iff j <= t.
 *   - LSE is the natural log of sum_j exp(s_tj) of the scaled scores.
 *   - layout [B, T, H, D] row-major for q/k/v/o/dO and their gradients;
 *     [B, Hq, T] for lse.  Query head h reads key/value head h / (Hq/Hkv).
 *
 * Every function works in double precision on double inputs (the caller
 * widens bf16 values exactly).  Only (batch, kv-head) groups whose entry in
 * `sel` is non-zero are computed; other outputs are left untouched, so a test
 * can check a sample of groups of a large problem exactly.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX4(b, t, h, d, T, H, D) ((((size_t)(b) * (T) + (t)) * (H) + (h)) * (D) + (d))

/* Rotation of one D-vector at position t, in place: pair i is (x[2i], x[2i+1])
 * (interleaved) or, with half != 0, (x[i], x[i + D/2]) (half-split).
 * dir = +1 applies R_t, dir = -1 applies R_t^T = R_{-t} (the adjoint used by
 * the backward pass: the rotation is orthogonal). */
static void rope_vec(double* x, int D, long t, double base, int dir, int half) {
  for (int i = 0; i < D / 2; i++) {
    double theta = pow(base, -2.0 * (double)i / (double)D);
    double ang = (double)t * theta;
    double c = cos(ang), s = sin(ang) * (double)dir;
    int i0 = half ? i : 2 * i, i1 = half ? i + D / 2 : 2 * i + 1;
    double x0 = x[i0], x1 = x[i1];
    x[i0] = x0 * c - x1 * s;
    x[i1] = x0 * s + x1 * c;
  }
}

/* out[b,t,h,:] = R_t x[b,t,h,:]  (dir=+1)  or  R_t^T x  (dir=-1). */
void oracle_rope(const double* x, double* out, int B, int T, int H, int D,
                 double base, int dir, int half) {
  size_t n = (size_t)B * T * H * D;
  memcpy(out, x, n * sizeof(double));
  for (int b = 0; b < B; b++)
    for (int t = 0; t < T; t++)
      for (int h = 0; h < H; h++)
        rope_vec(out + IDX4(b, t, h, 0, T, H, D), D, t, base, dir, half);
}

static double dot(const double* a, const double* b, int D) {
  double s = 0.0;
  for (int d = 0; d < D; d++) s += a[d] * b[d];
  return s;
}

/* Rotated copies of the queries of every head in kv-group g and of kv head g,
 * for batch b: qh[(hh*T + t)*D + d], kh[t*D + d]; vh and the upstream
 * gradient rows are gathered the same way for contiguous access. */
static void gather_group(const double* q, const double* k, const double* v,
                         const double* dout, int b, int g, int T, int Hq,
                         int Hkv, int D, double base, int half, double* qh, double* kh,
                         double* vh, double* doh) {
  int G = Hq / Hkv;
  for (int hh = 0; hh < G; hh++) {
    int h = g * G + hh;
    for (int t = 0; t < T; t++) {
      double* dst = qh + ((size_t)hh * T + t) * D;
      memcpy(dst, q + IDX4(b, t, h, 0, T, Hq, D), D * sizeof(double));
      rope_vec(dst, D, t, base, +1, half);
      if (doh)
        memcpy(doh + ((size_t)hh * T + t) * D, dout + IDX4(b, t, h, 0, T, Hq, D),
               D * sizeof(double));
    }
  }
  for (int t = 0; t < T; t++) {
    double* dk = kh + (size_t)t * D;
    memcpy(dk, k + IDX4(b, t, g, 0, T, Hkv, D), D * sizeof(double));
    rope_vec(dk, D, t, base, +1, half);
    memcpy(vh + (size_t)t * D, v + IDX4(b, t, g, 0, T, Hkv, D), D * sizeof(double));
  }
}

/* One query row of the forward pass: scores over the whole key range with the
 * causal mask applied explicitly, softmax with the row maximum subtracted,
 * then the probability-weighted sum of values.  s and p are length-T scratch.
 * Returns LSE_t; writes P into p (zero where masked) and O_t into o. */
static double fwd_row(const double* qt, const double* kh, const double* vh,
                      int t, int T, int D, double scale, double* s, double* p,
                      double* o) {
  double m = -INFINITY;
  for (int j = 0; j < T; j++) {
    s[j] = (j > t) ? -INFINITY : scale * dot(qt, kh + (size_t)j * D, D);
    if (s[j] > m) m = s[j];
  }
  double z = 0.0;
  for (int j = 0; j < T; j++) {
    p[j] = (j > t) ? 0.0 : exp(s[j] - m);
    z += p[j];
  }
  for (int j = 0; j < T; j++) p[j] /= z;
  for (int d = 0; d < D; d++) o[d] = 0.0;
  for (int j = 0; j < T; j++) {
    if (p[j] == 0.0) continue;
    const double* vj = vh + (size_t)j * D;
    for (int d = 0; d < D; d++) o[d] += p[j] * vj[d];
  }
  return m + log(z);
}

static int default_threads(int nthreads) {
#ifdef _OPENMP
  return nthreads > 0 ? nthreads : omp_get_max_threads();
#else
  (void)nthreads;
  return 1;
#endif
}

/* Forward: o [B,T,Hq,D], lse [B,Hq,T]. */
void oracle_attn_fwd(const double* q, const double* k, const double* v,
                     double* o, double* lse, int B, int T, int Hq, int Hkv,
                     int D, double base, int half, const unsigned char* sel,
                     int nthreads) {
  int G = Hq / Hkv;
  double scale = 1.0 / sqrt((double)D);
  int nt = default_threads(nthreads);
  double* qh = malloc(sizeof(double) * (size_t)G * T * D);
  double* kh = malloc(sizeof(double) * (size_t)T * D);
  double* vh = malloc(sizeof(double) * (size_t)T * D);
  for (int b = 0; b < B; b++)
    for (int g = 0; g < Hkv; g++) {
      if (sel && !sel[b * Hkv + g]) continue;
      gather_group(q, k, v, NULL, b, g, T, Hq, Hkv, D, base, half, qh, kh, vh, NULL);
#pragma omp parallel num_threads(nt)
      {
        double* s = malloc(sizeof(double) * T);
        double* p = malloc(sizeof(double) * T);
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < (long)G * T; r++) {
          int hh = (int)(r / T), t = (int)(r % T);
          int h = g * G + hh;
          double* ot = o + IDX4(b, t, h, 0, T, Hq, D);
          double l = fwd_row(qh + (size_t)r * D, kh, vh, t, T, D, scale, s, p, ot);
          lse[((size_t)b * Hq + h) * T + t] = l;
        }
        free(s);
        free(p);
      }
    }
  free(qh);
  free(kh);
  free(vh);
}

/* Backward, from the definition of each gradient (see the header comment for
 * the readings).  Given dO, for query row t of head h:
 *   dP_tj = dO_t . v_j,  D_t = sum_j P_tj dP_tj,  dS_tj = P_tj (dP_tj - D_t),
 *   dq_t  = R_t^T ( scale * sum_j dS_tj k^_j ),
 * and for key row j of kv head g (summing over the group's query heads, the
 * adjoint of repeating the key/value head across the group):
 *   dk_j  = R_j^T ( scale * sum_{h in group} sum_t dS_tj q^_t ),
 *   dv_j  = sum_{h in group} sum_t P_tj dO_t.
 * Pass 1 walks query rows (dq, and the per-row LSE_t and D_t); pass 2 walks
 * key rows and rebuilds P_tj = exp(s_tj - LSE_t) from the same scores.
 * Optional outputs: o, lse, delta ([B,Hq,T], the D_t above); pass NULL to skip.
 */
void oracle_attn_bwd(const double* q, const double* k, const double* v,
                     const double* dout, double* dq, double* dk, double* dv,
                     double* o, double* lse, double* delta, int B, int T,
                     int Hq, int Hkv, int D, double base, int half,
                     const unsigned char* sel, int nthreads) {
  int G = Hq / Hkv;
  double scale = 1.0 / sqrt((double)D);
  int nt = default_threads(nthreads);
  double* qh = malloc(sizeof(double) * (size_t)G * T * D);
  double* doh = malloc(sizeof(double) * (size_t)G * T * D);
  double* kh = malloc(sizeof(double) * (size_t)T * D);
  double* vh = malloc(sizeof(double) * (size_t)T * D);
  double* rl = malloc(sizeof(double) * (size_t)G * T); /* LSE_t per row */
  double* rd = malloc(sizeof(double) * (size_t)G * T); /* D_t per row */
  for (int b = 0; b < B; b++)
    for (int g = 0; g < Hkv; g++) {
      if (sel && !sel[b * Hkv + g]) continue;
      gather_group(q, k, v, dout, b, g, T, Hq, Hkv, D, base, half, qh, kh, vh, doh);
      /* pass 1: query rows */
#pragma omp parallel num_threads(nt)
      {
        double* s = malloc(sizeof(double) * T);
        double* p = malloc(sizeof(double) * T);
        double* ot = malloc(sizeof(double) * D);
        double* acc = malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 4)
        for (long r = 0; r < (long)G * T; r++) {
          int hh = (int)(r / T), t = (int)(r % T);
          int h = g * G + hh;
          const double* dot_ = doh + (size_t)r * D;
          double l = fwd_row(qh + (size_t)r * D, kh, vh, t, T, D, scale, s, p, ot);
          /* D_t from its definition: sum_j P_tj dP_tj */
          double dt = 0.0;
          for (int j = 0; j < T; j++)
            if (p[j] != 0.0) dt += p[j] * dot(dot_, vh + (size_t)j * D, D);
          for (int d = 0; d < D; d++) acc[d] = 0.0;
          for (int j = 0; j < T; j++) {
            if (p[j] == 0.0) continue;
            double dsj = p[j] * (dot(dot_, vh + (size_t)j * D, D) - dt);
            const double* kj = kh + (size_t)j * D;
            for (int d = 0; d < D; d++) acc[d] += dsj * kj[d];
          }
          for (int d = 0; d < D; d++) acc[d] *= scale;
          rope_vec(acc, D, t, base, -1, half);
          memcpy(dq + IDX4(b, t, h, 0, T, Hq, D), acc, D * sizeof(double));
          rl[r] = l;
          rd[r] = dt;
          if (o) memcpy(o + IDX4(b, t, h, 0, T, Hq, D), ot, D * sizeof(double));
          if (lse) lse[((size_t)b * Hq + h) * T + t] = l;
          if (delta) delta[((size_t)b * Hq + h) * T + t] = dt;
        }
        free(s);
        free(p);
        free(ot);
        free(acc);
      }
      /* pass 2: key rows */
#pragma omp parallel num_threads(nt)
      {
        double* ak = malloc(sizeof(double) * D);
        double* av = malloc(sizeof(double) * D);
#pragma omp for schedule(dynamic, 4)
        for (int j = 0; j < T; j++) {
          const double* kj = kh + (size_t)j * D;
          const double* vj = vh + (size_t)j * D;
          for (int d = 0; d < D; d++) ak[d] = av[d] = 0.0;
          for (int hh = 0; hh < G; hh++)
            for (int t = j; t < T; t++) { /* causal: only queries t >= j see key j */
              size_t r = (size_t)hh * T + t;
              const double* qt = qh + r * D;
              const double* dot_ = doh + r * D;
              double pij = exp(scale * dot(qt, kj, D) - rl[r]);
              double dsij = pij * (dot(dot_, vj, D) - rd[r]);
              for (int d = 0; d < D; d++) {
                ak[d] += dsij * qt[d];
                av[d] += pij * dot_[d];
              }
            }
          for (int d = 0; d < D; d++) ak[d] *= scale;
          rope_vec(ak, D, j, base, -1, half);
          memcpy(dk + IDX4(b, j, g, 0, T, Hkv, D), ak, D * sizeof(double));
          memcpy(dv + IDX4(b, j, g, 0, T, Hkv, D), av, D * sizeof(double));
        }
        free(ak);
        free(av);
      }
    }
  free(qh);
  free(doh);
  free(kh);
  free(vh);
  free(rl);
  free(rd);
}

int oracle_num_threads(void) { return default_threads(0); }
