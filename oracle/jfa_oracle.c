/*
 * jfa_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what jagged attention computes.  It exists
 * so that the CUDA path can be checked against something obviously correct; only
 * the tests, the smoke check and the benchmark's CPU-baseline leg may load it.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What is computed (sources are the four pages collected on jagged / block
 * attention with TLX):
 *   - Packed ("jagged") sequences addressed by an offsets array: sequence b holds
 *     rows [offsets[b], offsets[b+1]) of a [tokens, heads, dim] buffer
 *     ("Optimizing Jagged Flash Attention with TLX" commentary, section on why
 *     unequal lengths change the problem; the n1n.ai page's worked example with
 *     offsets [0, 128, 4224, 4736, 6784]).
 *   - Exact attention per sequence and head: s_ij = scale * q_i . k_j,
 *     P = row softmax(s), O = P V, and the log-sum-exp L = m + log(l) that the
 *     standard flash-attention loop stores for the backward pass ("TLX Block
 *     Attention" section 2.1, Listing 1).  The oracle evaluates the full score row
 *     and then the softmax; it does NOT use the online (running max / rescale)
 *     recurrence, so it checks a tiled kernel independently.
 *   - Broadcast-Q: one dense Q of Nq rows attends to every jagged K/V sequence;
 *     sequence b produces output rows b*Nq .. b*Nq+Nq-1 and the gradient of the
 *     shared Q is the sum over all sequences (commentary section on unequal
 *     lengths; aixai.ru summary, "What is Jagged Flash Attention").
 *   - Backward: dV = P^T dO, dP = dO V^T, Di = rowsum(P o dP), dS = P o (dP - Di),
 *     dQ = scale dS K, dK = scale dS^T Q ("TLX Block Attention" section 4; the
 *     aixai.ru summary counts five GEMMs per K/V block).  Di equals dO . O for the
 *     exact O; the oracle uses the exact form rowsum(P o dP).
 *   - Block-diagonal mode: every sequence is cut into blocks of `block` tokens
 *     (64 on the pages) and each block attends only within itself, with no
 *     log-sum-exp output ("TLX Block Attention" sections 1 and 2.1).
 *   - GQA: H query heads share Hkv key/value heads; query head h reads key/value
 *     head h / (H / Hkv) (the commentary's limits paragraph says GQA exists; the
 *     contiguous-group map is this code's reading).
 *   - Causal: key j is visible to query i iff j <= i within the sequence (reading;
 *     the pages do not define causal masking for the jagged kernel).
 *   - Sliding window: key j is visible to query i iff i - left <= j <= i + right
 *     within the sequence, a negative bound leaving its side open; causal
 *     attention is (left open, right 0).  The pages name windows among the
 *     variants the kernels keep (commentary, "performance and feature scope";
 *     aixai.ru summary, "MXFP8 and sparsity") without defining them; this
 *     two-sided local window is the reading.
 *
 * All inputs and outputs are fp64 arrays, row-major [rows, heads, dim].  Work is
 * split over threads by (sequence, head) units; nothing is blocked or reordered
 * beyond that.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* ------------------------------------------------------------------------- */
/* one attention segment, one head                                            */
/* ------------------------------------------------------------------------- */

static double dot(const double* a, const double* b, int n) {
  double s = 0.0;
  for (int d = 0; d < n; ++d) s += a[d] * b[d];
  return s;
}

/* Keys query row i may see: j in [*lo, *hi).  A negative left or right leaves
   that side open; causal attention is left < 0, right = 0. */
static void visible_range(int i, int nkeys, int left, int right, int* lo, int* hi) {
  int a = 0, e = nkeys;
  if (left >= 0 && i - left > a) a = i - left;
  if (right >= 0 && i + right + 1 < e) e = i + right + 1;
  *lo = a;
  *hi = e > a ? e : a;
}

/*
 * Forward for nrows queries against nkeys keys of one head.  Row i of Q sits at
 * q + i*qs; key j at k + j*ks (same for v); output row i at o + i*os.
 * p is scratch of nkeys doubles.  lse may be NULL.
 */
static void segment_fwd(const double* q, long qs, const double* k, const double* v, long ks,
                        int nrows, int nkeys, int D, double scale, int left, int right,
                        double* o, long os, double* lse, long lse_stride, double* p) {
  for (int i = 0; i < nrows; ++i) {
    int j0, n;
    visible_range(i, nkeys, left, right, &j0, &n);
    double* oi = o + (long)i * os;
    if (n == j0) {
      for (int d = 0; d < D; ++d) oi[d] = 0.0;
      if (lse) lse[(long)i * lse_stride] = -INFINITY;
      continue;
    }
    /* full score row, then its maximum */
    double m = -INFINITY;
    for (int j = j0; j < n; ++j) {
      p[j] = scale * dot(q + (long)i * qs, k + (long)j * ks, D);
      if (p[j] > m) m = p[j];
    }
    /* softmax normaliser */
    double l = 0.0;
    for (int j = j0; j < n; ++j) {
      p[j] = exp(p[j] - m);
      l += p[j];
    }
    /* O_i = sum_j P_ij V_j */
    for (int d = 0; d < D; ++d) oi[d] = 0.0;
    for (int j = j0; j < n; ++j) {
      const double pij = p[j] / l;
      const double* vj = v + (long)j * ks;
      for (int d = 0; d < D; ++d) oi[d] += pij * vj[d];
    }
    if (lse) lse[(long)i * lse_stride] = m + log(l);
  }
}

/*
 * Backward for one segment and one head.  Adds into dq (rows like q), dk and dv
 * (rows like k).  p and dp are scratch of nkeys doubles each.
 */
static void segment_bwd(const double* q, long qs, const double* k, const double* v, long ks,
                        const double* dout, long dos, int nrows, int nkeys, int D,
                        double scale, int left, int right, double* dq, long dqs, double* dk,
                        double* dv, long dks, double* p, double* dp) {
  for (int i = 0; i < nrows; ++i) {
    int j0, n;
    visible_range(i, nkeys, left, right, &j0, &n);
    if (n == j0) continue;
    const double* qi = q + (long)i * qs;
    const double* doi = dout + (long)i * dos;
    /* recompute the softmax row P_i */
    double m = -INFINITY;
    for (int j = j0; j < n; ++j) {
      p[j] = scale * dot(qi, k + (long)j * ks, D);
      if (p[j] > m) m = p[j];
    }
    double l = 0.0;
    for (int j = j0; j < n; ++j) {
      p[j] = exp(p[j] - m);
      l += p[j];
    }
    for (int j = j0; j < n; ++j) p[j] /= l;
    /* dP_ij = dO_i . V_j and Di = sum_j P_ij dP_ij */
    double di = 0.0;
    for (int j = j0; j < n; ++j) {
      dp[j] = dot(doi, v + (long)j * ks, D);
      di += p[j] * dp[j];
    }
    /* dS_ij = P_ij (dP_ij - Di); dQ_i += scale dS_ij K_j; dK_j += scale dS_ij Q_i;
       dV_j += P_ij dO_i */
    double* dqi = dq + (long)i * dqs;
    for (int j = j0; j < n; ++j) {
      const double ds = p[j] * (dp[j] - di);
      const double* kj = k + (long)j * ks;
      double* dkj = dk + (long)j * dks;
      double* dvj = dv + (long)j * dks;
      for (int d = 0; d < D; ++d) {
        dqi[d] += scale * ds * kj[d];
        dkj[d] += scale * ds * qi[d];
        dvj[d] += p[j] * doi[d];
      }
    }
  }
}

/* ------------------------------------------------------------------------- */
/* job description and a minimal thread pool                                  */
/* ------------------------------------------------------------------------- */

typedef struct {
  /* problem */
  const double *q, *k, *v, *dout;
  const int32_t* offsets;
  int batch, nq, H, Hkv, D, left, right, block; /* left, right: visible window (see visible_range) */
  double scale;
  const uint8_t* sel; /* [batch*H] or NULL: which (b, h) units to evaluate */
  double *o, *lse, *dq, *dk, *dv;
  /* work split */
  int kind;        /* 0 fwd, 1 bwd self, 2 bwd broadcast, 3 block fwd, 4 block bwd */
  long n_units;
  long next;       /* atomic counter */
  int max_len;
  int n_chunks;    /* broadcast backward: sequences are grouped into chunks */
  double* dq_part; /* broadcast backward: [n_chunks*H, nq, D] partial sums */
} job_t;

static int seq_len(const job_t* J, int b) { return J->offsets[b + 1] - J->offsets[b]; }
static int unit_selected(const job_t* J, int b, int h) {
  return J->sel == NULL || J->sel[(long)b * J->H + h] != 0;
}

static void run_unit(job_t* J, long u, double* p, double* dp) {
  const int H = J->H, Hkv = J->Hkv, D = J->D, G = H / Hkv;
  const long qs = (long)H * D, ks = (long)Hkv * D;
  if (J->kind == 0 || J->kind == 3) {
    /* unit = (b, h) */
    const int b = (int)(u / H), h = (int)(u % H), g = h / G;
    if (!unit_selected(J, b, h)) return;
    const int L = seq_len(J, b);
    const long t0 = J->offsets[b];
    const double* kb = J->k + t0 * ks + (long)g * D;
    const double* vb = J->v + t0 * ks + (long)g * D;
    if (J->kind == 3) {
      for (int s = 0; s < L; s += J->block) {
        const int n = (L - s < J->block) ? L - s : J->block;
        segment_fwd(J->q + (t0 + s) * qs + (long)h * D, qs, kb + (long)s * ks, vb + (long)s * ks, ks,
                    n, n, D, J->scale, -1, -1, J->o + (t0 + s) * qs + (long)h * D, qs, NULL, 0, p);
      }
    } else if (J->nq > 0) {
      /* broadcast-Q: shared Q rows, output rows b*nq .. */
      const long r0 = (long)b * J->nq;
      const long total_rows = (long)J->batch * J->nq;
      segment_fwd(J->q + (long)h * D, qs, kb, vb, ks, J->nq, L, D, J->scale, -1, -1,
                  J->o + r0 * qs + (long)h * D, qs, J->lse ? J->lse + (long)h * total_rows + r0 : NULL, 1, p);
    } else {
      const long total_rows = J->offsets[J->batch];
      segment_fwd(J->q + t0 * qs + (long)h * D, qs, kb, vb, ks, L, L, D, J->scale, J->left, J->right,
                  J->o + t0 * qs + (long)h * D, qs, J->lse ? J->lse + (long)h * total_rows + t0 : NULL, 1, p);
    }
    return;
  }
  if (J->kind == 1 || J->kind == 4) {
    /* unit = (b, g): every query head of group g adds into dK/dV of head g */
    const int b = (int)(u / Hkv), g = (int)(u % Hkv);
    const int L = seq_len(J, b);
    const long t0 = J->offsets[b];
    for (int h = g * G; h < (g + 1) * G; ++h) {
      if (!unit_selected(J, b, h)) continue;
      const int step = (J->kind == 4) ? J->block : (L > 0 ? L : 1);
      for (int s = 0; s < L; s += step) {
        const int n = (L - s < step) ? L - s : step;
        const long r = t0 + s;
        segment_bwd(J->q + r * qs + (long)h * D, qs, J->k + r * ks + (long)g * D, J->v + r * ks + (long)g * D, ks,
                    J->dout + r * qs + (long)h * D, qs, n, n, D, J->scale, J->kind == 1 ? J->left : -1,
                    J->kind == 1 ? J->right : -1,
                    J->dq + r * qs + (long)h * D, qs, J->dk + r * ks + (long)g * D, J->dv + r * ks + (long)g * D,
                    ks, p, dp);
      }
    }
    return;
  }
  /* kind 2: broadcast backward; unit = (chunk, g) over the sequences of the chunk.
     dQ of the shared Q goes to this unit's own partial buffer. */
  {
    const int c = (int)(u / Hkv), g = (int)(u % Hkv);
    const int b0 = (int)((long)c * J->batch / J->n_chunks);
    const int b1 = (int)((long)(c + 1) * J->batch / J->n_chunks);
    const long nq = J->nq;
    for (int h = g * G; h < (g + 1) * G; ++h) {
      double* part = J->dq_part + ((long)c * H + h) * nq * D;
      for (int b = b0; b < b1; ++b) {
        if (!unit_selected(J, b, h)) continue;
        const int L = seq_len(J, b);
        const long t0 = J->offsets[b];
        segment_bwd(J->q + (long)h * D, qs, J->k + t0 * ks + (long)g * D, J->v + t0 * ks + (long)g * D, ks,
                    J->dout + (long)b * nq * qs + (long)h * D, qs, (int)nq, L, D, J->scale, -1, -1,
                    part, D, J->dk + t0 * ks + (long)g * D, J->dv + t0 * ks + (long)g * D, ks, p, dp);
      }
    }
  }
}

static void* worker(void* arg) {
  job_t* J = (job_t*)arg;
  const int n = J->max_len > J->block ? J->max_len : J->block;
  double* p = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  double* dp = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
  for (;;) {
    const long u = __atomic_fetch_add(&J->next, 1, __ATOMIC_RELAXED);
    if (u >= J->n_units) break;
    run_unit(J, u, p, dp);
  }
  free(p);
  free(dp);
  return NULL;
}

static int run_job(job_t* J, int nthreads) {
  if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
  if (nthreads < 1) nthreads = 1;
  if (nthreads > J->n_units) nthreads = (int)(J->n_units > 0 ? J->n_units : 1);
  J->next = 0;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
  int started = 0;
  for (int t = 0; t < nthreads; ++t)
    if (pthread_create(&th[t], NULL, worker, J) == 0) ++started;
  if (started == 0) worker(J);
  for (int t = 0; t < started; ++t) pthread_join(th[t], NULL);
  free(th);
  return started > 0 ? started : 1;
}

static int check_common(const int32_t* offsets, int batch, int H, int Hkv, int D, int* max_len) {
  if (batch < 0 || H <= 0 || Hkv <= 0 || D <= 0 || H % Hkv != 0 || offsets == NULL) return -1;
  if (offsets[0] != 0) return -2;
  int ml = 0;
  for (int b = 0; b < batch; ++b) {
    const int L = offsets[b + 1] - offsets[b];
    if (L < 0) return -2;
    if (L > ml) ml = L;
  }
  *max_len = ml;
  return 0;
}

/* ------------------------------------------------------------------------- */
/* exported entry points (called from Python through ctypes)                  */
/* ------------------------------------------------------------------------- */

/*
 * Forward.  nq == 0: self-attention, q/o [T,H,D], k/v [T,Hkv,D], lse [H,T].
 * nq > 0: broadcast-Q, q [nq,H,D], o [batch*nq,H,D], lse [H,batch*nq]; causal must be 0.
 * sel: optional [batch*H] bytes choosing which (b,h) units to evaluate.
 * Returns the number of threads used, or a negative error.
 */
int oracle_attn_fwd_window(const double* q, const double* k, const double* v, const int32_t* offsets,
                           int batch, int nq, int H, int Hkv, int D, double scale, int left, int right,
                           const uint8_t* sel, double* o, double* lse, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  if (check_common(offsets, batch, H, Hkv, D, &J.max_len)) return -1;
  if (nq > 0 && (left >= 0 || right >= 0)) return -1;
  J.q = q; J.k = k; J.v = v; J.offsets = offsets; J.batch = batch; J.nq = nq;
  J.H = H; J.Hkv = Hkv; J.D = D; J.scale = scale; J.left = left; J.right = right; J.sel = sel;
  J.o = o; J.lse = lse; J.kind = 0; J.n_units = (long)batch * H; J.block = 1;
  return run_job(&J, nthreads);
}

/* The same without a window, or causal (left open, right 0). */
int oracle_attn_fwd(const double* q, const double* k, const double* v, const int32_t* offsets,
                    int batch, int nq, int H, int Hkv, int D, double scale, int causal,
                    const uint8_t* sel, double* o, double* lse, int nthreads) {
  return oracle_attn_fwd_window(q, k, v, offsets, batch, nq, H, Hkv, D, scale, -1, causal ? 0 : -1, sel, o, lse,
                                nthreads);
}

/*
 * Backward.  Inputs as in the forward plus dout (shaped like o).  Outputs dq
 * (shaped like q), dk and dv (shaped like k); all three are overwritten.
 * Broadcast mode sums the shared-Q gradient over all sequences.
 */
int oracle_attn_bwd_window(const double* q, const double* k, const double* v, const double* dout,
                           const int32_t* offsets, int batch, int nq, int H, int Hkv, int D, double scale,
                           int left, int right, const uint8_t* sel, double* dq, double* dk, double* dv,
                           int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  if (check_common(offsets, batch, H, Hkv, D, &J.max_len)) return -1;
  if (nq > 0 && (left >= 0 || right >= 0)) return -1;
  const long T = offsets[batch];
  J.q = q; J.k = k; J.v = v; J.dout = dout; J.offsets = offsets; J.batch = batch; J.nq = nq;
  J.H = H; J.Hkv = Hkv; J.D = D; J.scale = scale; J.left = left; J.right = right; J.sel = sel;
  J.dq = dq; J.dk = dk; J.dv = dv; J.block = 1;
  memset(dk, 0, sizeof(double) * (size_t)(T * Hkv * D));
  memset(dv, 0, sizeof(double) * (size_t)(T * Hkv * D));
  if (nq == 0) {
    memset(dq, 0, sizeof(double) * (size_t)(T * H * D));
    J.kind = 1;
    J.n_units = (long)batch * Hkv;
    return run_job(&J, nthreads);
  }
  /* broadcast: per-chunk partial dQ, summed afterwards in chunk order */
  J.kind = 2;
  J.n_chunks = batch < 64 ? (batch > 0 ? batch : 1) : 64;
  J.n_units = (long)J.n_chunks * Hkv;
  const size_t part = (size_t)nq * D;
  J.dq_part = (double*)calloc((size_t)J.n_chunks * H * part, sizeof(double));
  if (!J.dq_part) return -3;
  const int used = run_job(&J, nthreads);
  for (int h = 0; h < H; ++h)
    for (long i = 0; i < nq; ++i)
      for (int d = 0; d < D; ++d) {
        double s = 0.0;
        for (int c = 0; c < J.n_chunks; ++c) s += J.dq_part[((size_t)c * H + h) * part + (size_t)i * D + d];
        dq[(i * H + h) * D + d] = s;
      }
  free(J.dq_part);
  return used;
}

/* The same without a window, or causal (left open, right 0). */
int oracle_attn_bwd(const double* q, const double* k, const double* v, const double* dout,
                    const int32_t* offsets, int batch, int nq, int H, int Hkv, int D, double scale,
                    int causal, const uint8_t* sel, double* dq, double* dk, double* dv, int nthreads) {
  return oracle_attn_bwd_window(q, k, v, dout, offsets, batch, nq, H, Hkv, D, scale, -1, causal ? 0 : -1, sel,
                                dq, dk, dv, nthreads);
}

/* Block-diagonal forward: blocks of `block` tokens inside each sequence; no LSE. */
int oracle_block_fwd(const double* q, const double* k, const double* v, const int32_t* offsets,
                     int batch, int H, int D, double scale, int block, const uint8_t* sel,
                     double* o, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  if (block <= 0 || check_common(offsets, batch, H, H, D, &J.max_len)) return -1;
  J.q = q; J.k = k; J.v = v; J.offsets = offsets; J.batch = batch; J.H = H; J.Hkv = H; J.D = D;
  J.scale = scale; J.block = block; J.sel = sel; J.o = o; J.kind = 3; J.n_units = (long)batch * H;
  return run_job(&J, nthreads);
}

/* Block-diagonal backward. */
int oracle_block_bwd(const double* q, const double* k, const double* v, const double* dout,
                     const int32_t* offsets, int batch, int H, int D, double scale, int block,
                     const uint8_t* sel, double* dq, double* dk, double* dv, int nthreads) {
  job_t J;
  memset(&J, 0, sizeof J);
  if (block <= 0 || check_common(offsets, batch, H, H, D, &J.max_len)) return -1;
  const long T = offsets[batch];
  J.q = q; J.k = k; J.v = v; J.dout = dout; J.offsets = offsets; J.batch = batch; J.H = H; J.Hkv = H;
  J.D = D; J.scale = scale; J.block = block; J.sel = sel; J.dq = dq; J.dk = dk; J.dv = dv; J.kind = 4;
  J.n_units = (long)batch * H;
  memset(dq, 0, sizeof(double) * (size_t)(T * H * D));
  memset(dk, 0, sizeof(double) * (size_t)(T * H * D));
  memset(dv, 0, sizeof(double) * (size_t)(T * H * D));
  return run_job(&J, nthreads);
}
