/*
 * KDA oracle: TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, sequential fp64 CPU implementation of Kimi Delta Attention
 * (KDA), token by token.  It exists to check the CUDA library; only the test
 * suite, the smoke check and the benchmark's CPU-baseline leg load it.  It
 * shares no code, header or constant with the CUDA path.
 *
 * What it computes (per sequence, per head; S is dk x dv, row index = key
 * channel i, column index = value channel j):
 *
 *   gate       g_t[i] = gmin * sigmoid(exp(A_h) * z_t[i]),  gmin = -5
 *              "Kimi K3 Technical Report - Open Frontier Intelligence",
 *              Key claims and Method (sec. 2.1.1, Fig. 3): the scaled-sigmoid
 *              log-decay bounded below at gmin = -5 with a learnable per-head A.
 *              The decay is channel-wise (one value per key channel), the
 *              reading of sec. 2.1.2 on that page ("matching KDA's new gating",
 *              channel-wise full-rank gate).
 *   recurrence S_t = (I - b_t k_t k_t^T) Diag(exp(g_t)) S_{t-1} + b_t k_t v_t^T
 *              o_t = S_t^T q_t
 *              a delta-rule write into a fixed-size running state that replaces
 *              the KV cache ("How a Frontier Model Gets Built, Read from the
 *              Kimi K3 Report", TL;DR and Technical Details: Delta Attention
 *              with a fixed-size running state).  The pages do not print the
 *              update; this gated delta rule is the reading adopted.
 *
 * The product form above is evaluated in its expanded, algebraically equal
 * order: decay the state, read the decayed state with the key (p = S^T k),
 * write b*k*(v - p)^T, read the output with the query.  With erase = 0 the
 * p term is dropped (S_t = Diag(exp(g_t)) S_{t-1} + b_t k_t v_t^T), the gated
 * linear attention reading used only by the oracle's own pins.
 *
 * Layouts (row-major, C order):
 *   q, k, z  [total_tokens, H, dk]      v, o  [total_tokens, H, dv]
 *   beta     [total_tokens, H]          A     [H]
 *   states   [n, H, dk, dv]             cu_seqlens [n_seq + 1] (token offsets)
 *   snapshots [snap_offsets[n_seq], H, dk, dv]: snapshot j (j = 1..floor(L/chunk))
 *   of sequence s is the state after its first j*chunk tokens, stored at row
 *   snap_offsets[s] + j - 1.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Log-decay of one channel: g = gmin * sigmoid(exp(A) * z).
 * sigmoid(x) = 1 / (1 + exp(-x)); x = +inf gives 1, x = -inf gives 0. */
static double gate(double gmin, double A_h, double z) {
  const double x = exp(A_h) * z;
  return gmin / (1.0 + exp(-x));
}

/* One token of the recurrence on one (sequence, head) state. */
static void token_step(double *S, int dk, int dv, const double *q,
                       const double *k, const double *v, const double *z,
                       double b, double A_h, double gmin, int erase, double *o,
                       double *p) {
  /* decay: S <- Diag(exp(g)) S */
  for (int i = 0; i < dk; ++i) {
    const double a = exp(gate(gmin, A_h, z[i]));
    for (int j = 0; j < dv; ++j) S[(size_t)i * dv + j] *= a;
  }
  /* erase read-out: p = S^T k */
  for (int j = 0; j < dv; ++j) p[j] = 0.0;
  if (erase) {
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) p[j] += S[(size_t)i * dv + j] * k[i];
  }
  /* write: S <- S + b k (v - p)^T  ==  (I - b k k^T) S + b k v^T */
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j)
      S[(size_t)i * dv + j] += b * k[i] * (v[j] - p[j]);
  /* output: o = S^T q */
  for (int j = 0; j < dv; ++j) o[j] = 0.0;
  for (int i = 0; i < dk; ++i)
    for (int j = 0; j < dv; ++j) o[j] += S[(size_t)i * dv + j] * q[i];
}

/* Gate values for an array: g[t*H*dk + h*dk + i] for z of layout [T, H, dk]. */
void kda_ref_gate(const double *z, const double *A, double gmin, int64_t T,
                  int H, int dk, double *g) {
  for (int64_t t = 0; t < T; ++t)
    for (int h = 0; h < H; ++h)
      for (int i = 0; i < dk; ++i) {
        const size_t x = ((size_t)t * H + h) * dk + i;
        g[x] = gate(gmin, A[h], z[x]);
      }
}

int kda_ref_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Prefill over packed sequences.  S0, S_final, snaps and snap_offsets may be
 * NULL (S0 NULL = zero state).  chunk sets the snapshot spacing only; the
 * oracle itself is purely sequential.  Returns 0, or -1 on a bad argument. */
int kda_ref_prefill(const double *q, const double *k, const double *v,
                    const double *z, const double *beta, const double *A,
                    double gmin, const int64_t *cu_seqlens, int n_seq, int H,
                    int dk, int dv, int chunk, const double *S0, double *o,
                    double *S_final, double *snaps, const int64_t *snap_offsets,
                    int erase) {
  if (!q || !k || !v || !z || !beta || !A || !cu_seqlens || !o) return -1;
  if (n_seq < 0 || H <= 0 || dk <= 0 || dv <= 0 || chunk <= 0) return -1;
  if (snaps && !snap_offsets) return -1;
  const size_t sz = (size_t)dk * dv;
  const long long pairs = (long long)n_seq * H;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (long long ph = 0; ph < pairs; ++ph) {
    const int s = (int)(ph / H), h = (int)(ph % H);
    const int64_t t0 = cu_seqlens[s], t1 = cu_seqlens[s + 1];
    if (t1 < t0) { bad = 1; continue; }
    double *S = (double *)malloc(sz * sizeof(double));
    double *p = (double *)malloc((size_t)dv * sizeof(double));
    if (!S || !p) { free(S); free(p); bad = 1; continue; }
    if (S0) memcpy(S, S0 + ((size_t)s * H + h) * sz, sz * sizeof(double));
    else memset(S, 0, sz * sizeof(double));
    for (int64_t t = t0; t < t1; ++t) {
      const size_t xk = ((size_t)t * H + h) * dk, xv = ((size_t)t * H + h) * dv;
      token_step(S, dk, dv, q + xk, k + xk, v + xv, z + xk,
                 beta[(size_t)t * H + h], A[h], gmin, erase, o + xv, p);
      const int64_t n_done = t - t0 + 1;
      if (snaps && n_done % chunk == 0) {
        const int64_t row = snap_offsets[s] + n_done / chunk - 1;
        memcpy(snaps + ((size_t)row * H + h) * sz, S, sz * sizeof(double));
      }
    }
    if (S_final) memcpy(S_final + ((size_t)s * H + h) * sz, S, sz * sizeof(double));
    free(S);
    free(p);
  }
  return bad ? -1 : 0;
}

/* One decode step for n resident states [n, H, dk, dv], updated in place.
 * Inputs are one token per sequence: q, k, z [n, H, dk]; v, o [n, H, dv];
 * beta [n, H]. */
int kda_ref_decode_step(const double *q, const double *k, const double *v,
                        const double *z, const double *beta, const double *A,
                        double gmin, double *state, int n, int H, int dk,
                        int dv, double *o) {
  if (!q || !k || !v || !z || !beta || !A || !state || !o) return -1;
  if (n < 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
  const size_t sz = (size_t)dk * dv;
  const long long pairs = (long long)n * H;
  int bad = 0;
#pragma omp parallel for schedule(static) reduction(| : bad)
  for (long long ph = 0; ph < pairs; ++ph) {
    double *p = (double *)malloc((size_t)dv * sizeof(double));
    if (!p) { bad = 1; continue; }
    const int h = (int)(ph % H);
    token_step(state + (size_t)ph * sz, dk, dv, q + (size_t)ph * dk,
               k + (size_t)ph * dk, v + (size_t)ph * dv, z + (size_t)ph * dk,
               beta[ph], A[h], gmin, 1, o + (size_t)ph * dv, p);
    free(p);
  }
  return bad ? -1 : 0;
}
