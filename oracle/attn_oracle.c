/*
 * attn_oracle.c -- plain fp64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the correctness reference that the
 * GPU library is checked against.  Nothing in the product path may include,
 * link or call it: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg load it.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes, and where that is defined:
 *
 *   Standard attention, written out from its definition (page "突破单卡显存极限：
 *   FlashAttention-2技术解析与实战指南", section 1, the pseudocode
 *   "S = Q @ K.T ; P = softmax(S) ; return P @ V"), with the scale 1/sqrt(d_k)
 *   applied to the scores before the softmax (page "Flash Attention V2大模型时代
 *   的算力救星", section 4.2, the call flash_attention(q, k, v,
 *   softmax_scale=1.0/sqrt(d_k), ..., causal=...)):
 *
 *     s_rj  = scale * <q_r, k_j>              (j > r removed when causal)
 *     P_rj  = exp(s_rj) / sum_j exp(s_rj)
 *     O_r   = sum_j P_rj v_j
 *     LSE_r = log sum_j exp(s_rj)             (natural log)
 *
 *   The pages state that the tiled method gives exactly this result, not an
 *   approximation (page "FlashAttention-2：GPU利用率从50%干到90%，同一个作者的自我
 *   进化", section "数据说话", the sentence on identical output; page
 *   "突破单卡显存极限", section 2.1, the remark that the final result agrees with
 *   the full computation).  So the oracle is the definition, materialising one
 *   full score row at a time in fp64; it does no tiling and no online softmax.
 *
 *   The backward pass is not written out on the pages beyond "recompute in the
 *   backward pass instead of storing" (page "突破单卡显存极限", section 1 and
 *   section 2.2).  The oracle takes the plain calculus of the definition above
 *   for the loss L = sum(O * dO):
 *     dV_j  = sum_r P_rj dO_r
 *     dP_rj = <dO_r, v_j>
 *     D_r   = sum_j P_rj dP_rj          (the definition, not dO_r . O_r)
 *     dS_rj = P_rj (dP_rj - D_r)
 *     dQ_r  = scale * sum_j dS_rj k_j
 *     dK_j  = scale * sum_r dS_rj q_r
 *
 *   A second routine, oracle_online_fwd, follows the blockwise softmax
 *   recurrence of page "突破单卡显存极限", section 2.1 (m, l, m_j, f_j, l_j,
 *   m_new, l_new, f_j rescale) in the page's own order, with the two steps that
 *   the page leaves out made explicit (the assignment m <- m_new, l <- l_new
 *   and the rescaled output accumulator).  It exists only so that a test can
 *   check that the blockwise recurrence equals the full softmax.
 *
 *   ALiBi (page "FlashAttention技术解析：如何让GPT训练速度提升5-9倍", section 4.1,
 *   which names Attention with Linear Biases for long contexts and gives no
 *   formula): every routine but the blockwise one takes a per-head slope
 *   `alibi` (0 = none) and adds the linear bias -alibi * |pos(r) - j| to the
 *   scaled score s_rj, pos(r) being the position of query row r.  The bias
 *   is a constant of the inputs, so the backward formulas are unchanged.
 *
 *   Block-sparse masks (page "FlashAttention技术解析：如何让GPT训练速度提升5-9倍",
 *   section 5.2, names Block-Sparse FlashAttention): oracle_fwd and oracle_bwd
 *   take an optional per-head mask over 128 x 128 blocks, bmask[qb * nb + kb]
 *   for query block qb = r / 128 and key block kb = j / 128 (nb blocks per
 *   side); a zero entry removes those scores, like the causal mask.  A row
 *   left with no visible key has O = 0 and LSE = -inf and takes no part in
 *   the backward.
 *
 *   Dropout (page "Flash Attention V2大模型时代的算力救星", section 4.2, the
 *   call's dropout_p argument; page "FlashAttention-2：GPU利用率从50%干到90%",
 *   improvement 2, which counts dropout among the non-matmul operations done
 *   inside the kernel): oracle_fwd and oracle_bwd take an optional dropout of
 *   the attention probabilities.  Each P_rj is kept with probability
 *   q = t / 256 and then multiplied by 1 / q, or set to 0 ("inverted"
 *   dropout, so E[O] is the output without dropout):
 *     O_r   = sum_j Z_rj P_rj v_j / q            (Z_rj = 1 if kept, else 0)
 *     LSE_r = log sum_j exp(s_rj)                (before dropout)
 *   and the calculus of the backward, with P_rj replaced where it multiplies
 *   v_j:
 *     dV_j  = sum_r (Z_rj P_rj / q) dO_r
 *     dP_rj = Z_rj <dO_r, v_j> / q
 *     D_r   = sum_j P_rj dP_rj ;  dS_rj = P_rj (dP_rj - D_r) as above.
 *   The pages name no random number generator.  The decisions Z_rj come from
 *   the counter-based generator Philox4x32-10 of Salmon, Moraes, Dror and
 *   Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC 2011): key
 *   (low, high 32 bits of a 64-bit seed), counter (r, j / 16, head, offset);
 *   byte j % 16 of its 16 output bytes (word (j % 16) / 4, least significant
 *   byte first) decides key j: kept iff byte < t, with the threshold
 *   t = floor(256 (1 - p) + 1/2) for a dropout probability p.  The rounds
 *   are written once (a macro) for 32- and 64-bit words, the latter being
 *   Philox4x64-10.
 *
 *   A third routine, oracle_decode_fwd, is the same definition for Nq query
 *   rows against Nk keys (decoding with a key/value cache: page "FlashAttention
 *   技术解析：如何让GPT训练速度提升5-9倍", section 4.1 on the KV cache, and page
 *   "突破单卡显存极限", section 3.2 on vLLM inference).  The query rows are the
 *   last Nq positions of the sequence, so under the causal mask query i
 *   (0-based) sees keys j <= Nk - Nq + i, the same rows as the last Nq rows of
 *   a full Nk x Nk causal attention.
 *
 * Layout: every routine works on ONE attention head.  q, k, v, dO are
 * row-major [N][d] fp64 arrays (row n, column c at n*d + c).  The caller
 * slices heads out of [B,N,H,d] tensors.  Optional index lists select which
 * query rows (outputs O, LSE, dQ) and which key rows (dK, dV) are produced;
 * a NULL list means all rows, in order.
 *
 * Threads: query rows are split into contiguous ranges, one per thread
 * (pthreads).  Per-thread partial dK/dV sums are added in thread order, so the
 * result does not depend on scheduling.
 */
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL -1
#define ORACLE_ENOMEM -2

static int oracle_threads(int requested, int work) {
  int n = requested;
  if (n <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    n = c > 0 ? (int)c : 1;
  }
  if (n > work) n = work;
  if (n < 1) n = 1;
  return n;
}

int oracle_default_threads(void) { return oracle_threads(0, 1 << 30); }

/* ------------------------------------------------------------------------ */
/* Philox (Salmon et al., SC 2011, section 3.2): four words x0..x3, two key   */
/* words; each of R rounds multiplies x0 and x2 by the constants M0, M1 into  */
/* double-width products and forms                                            */
/*   (hi(M1 x2) ^ x1 ^ k0,  lo(M1 x2),  hi(M0 x0) ^ x3 ^ k1,  lo(M0 x0))      */
/* then bumps the key by the Weyl constants (W0, W1).  One body, two widths.  */
/* ------------------------------------------------------------------------ */
#define PHILOX_BODY(T, WIDE, BITS, M0, M1, W0, W1)                            \
  T x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];                       \
  T k0 = key[0], k1 = key[1];                                                 \
  for (int round = 0; round < 10; ++round) {                                  \
    WIDE p0 = (WIDE)(M0) * x0, p1 = (WIDE)(M1) * x2;                          \
    T hi0 = (T)(p0 >> (BITS)), lo0 = (T)p0;                                   \
    T hi1 = (T)(p1 >> (BITS)), lo1 = (T)p1;                                   \
    x0 = hi1 ^ x1 ^ k0;                                                       \
    x1 = lo1;                                                                 \
    x2 = hi0 ^ x3 ^ k1;                                                       \
    x3 = lo0;                                                                 \
    k0 += (W0);                                                               \
    k1 += (W1);                                                               \
  }                                                                           \
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;

void oracle_philox4x32(const unsigned int* ctr, const unsigned int* key,
                       unsigned int* out) {
  PHILOX_BODY(unsigned int, unsigned long long, 32, 0xD2511F53u, 0xCD9E8D57u,
              0x9E3779B9u, 0xBB67AE85u)
}

void oracle_philox4x64(const unsigned long long* ctr,
                       const unsigned long long* key, unsigned long long* out) {
  PHILOX_BODY(unsigned long long, unsigned __int128, 64, 0xD2E7470EE14C6C93ull,
              0xCA5A826395121157ull, 0x9E3779B97F4A7C15ull,
              0xBB67AE8584CAA73Bull)
}

/* Keep threshold for dropout probability p: t = floor(256 (1 - p) + 1/2),
 * kept iff byte < t; -1 for p outside [0, 1) or a threshold of 0. */
int oracle_dropout_threshold(double p) {
  if (!(p >= 0.0 && p < 1.0)) return -1;
  int t = (int)floor(256.0 * (1.0 - p) + 0.5);
  return t >= 1 ? t : -1;
}

typedef struct {
  int t;                  /* keep threshold 1..256 (256 keeps every score) */
  unsigned long long seed;
  unsigned int offset;
  unsigned int head;
} dropout_spec;

/* Z_rj: 1 if score (r, j) is kept. */
static int dropout_keep(const dropout_spec* dr, int r, int j) {
  unsigned int ctr[4] = {(unsigned int)r, (unsigned int)(j / 16), dr->head, dr->offset};
  unsigned int key[2] = {(unsigned int)(dr->seed & 0xFFFFFFFFull),
                         (unsigned int)(dr->seed >> 32)};
  unsigned int x[4];
  oracle_philox4x32(ctr, key, x);
  int b = j % 16;
  unsigned int byte = (x[b / 4] >> (8 * (b % 4))) & 0xFFu;
  return byte < (unsigned int)dr->t;
}

int oracle_dropout_keep(unsigned long long seed, unsigned int offset,
                        unsigned int head, int r, int j, int t) {
  dropout_spec dr = {t, seed, offset, head};
  return dropout_keep(&dr, r, j);
}

/* ------------------------------------------------------------------------ */
/* One score row: s_j = scale * <q_r, k_j> for j < ncols, P_rj = softmax.     */
/* ncols = r + 1 when causal (keys after r are removed), N otherwise.         */
/* Writes p[0..ncols) and returns LSE_r.                                      */
/* ------------------------------------------------------------------------ */
static double softmax_row(const double* q, const double* k, int N, int d,
                          double scale, double alibi, int causal,
                          const unsigned char* bmask, int nb, int r,
                          double* p, int* ncols_out) {
  int ncols = causal ? r + 1 : N;
  const double* qr = q + (size_t)r * d;
  double mx = -INFINITY;
  for (int j = 0; j < ncols; ++j) {
    if (bmask && !bmask[(size_t)(r / 128) * nb + j / 128]) {
      p[j] = -INFINITY; /* block removed by the sparse mask */
      continue;
    }
    const double* kj = k + (size_t)j * d;
    double s = 0.0;
    for (int c = 0; c < d; ++c) s += qr[c] * kj[c];
    s *= scale;
    s -= alibi * fabs((double)(r - j));
    p[j] = s;
    if (s > mx) mx = s;
  }
  *ncols_out = ncols;
  if (mx == -INFINITY) { /* no visible key: P = 0, O = 0, LSE = -inf */
    for (int j = 0; j < ncols; ++j) p[j] = 0.0;
    return -INFINITY;
  }
  /* exp(s - mx) keeps the sum finite; the row max is only a shift. */
  double z = 0.0;
  for (int j = 0; j < ncols; ++j) {
    p[j] = exp(p[j] - mx);
    z += p[j];
  }
  for (int j = 0; j < ncols; ++j) p[j] /= z;
  return mx + log(z);
}

/* ------------------------------------------------------------------------ */
/* Forward                                                                    */
/* ------------------------------------------------------------------------ */
typedef struct {
  const double *q, *k, *v;
  int N, d, causal;
  double scale, alibi;
  const unsigned char* bmask;
  int nb;
  const dropout_spec* dr; /* NULL: no dropout */
  const int* rows;
  int r0, r1; /* range in the output row list */
  double *o, *lse;
} fwd_job;

static void* fwd_worker(void* arg) {
  fwd_job* J = (fwd_job*)arg;
  double* p = (double*)malloc(sizeof(double) * (size_t)J->N);
  if (!p) return (void*)1;
  for (int i = J->r0; i < J->r1; ++i) {
    int r = J->rows ? J->rows[i] : i;
    int ncols;
    double lse = softmax_row(J->q, J->k, J->N, J->d, J->scale, J->alibi,
                             J->causal, J->bmask, J->nb, r, p, &ncols);
    double* orow = J->o + (size_t)i * J->d;
    for (int c = 0; c < J->d; ++c) orow[c] = 0.0;
    for (int j = 0; j < ncols; ++j) {
      double pj = p[j];
      if (J->dr) pj = dropout_keep(J->dr, r, j) ? pj * (256.0 / J->dr->t) : 0.0;
      const double* vj = J->v + (size_t)j * J->d;
      for (int c = 0; c < J->d; ++c) orow[c] += pj * vj[c];
    }
    if (J->lse) J->lse[i] = lse;
  }
  free(p);
  return NULL;
}

/* O[nrows][d] and LSE[nrows] for the query rows listed in `rows`
 * (NULL: all N rows, nrows must equal N). */
int oracle_fwd(const double* q, const double* k, const double* v, int N, int d,
               double scale, double alibi, int causal,
               const unsigned char* bmask, int drop_t, unsigned long long seed,
               unsigned int offset, unsigned int head, const int* rows,
               int nrows, double* o, double* lse, int nthreads) {
  const int nb = (N + 127) / 128;
  if (!q || !k || !v || !o || N < 1 || d < 1 || nrows < 0) return ORACLE_EINVAL;
  if (drop_t < 1 || drop_t > 256) return ORACLE_EINVAL;
  dropout_spec drs = {drop_t, seed, offset, head};
  const dropout_spec* dr = drop_t < 256 ? &drs : NULL;
  if (!rows && nrows != N) return ORACLE_EINVAL;
  if (rows)
    for (int i = 0; i < nrows; ++i)
      if (rows[i] < 0 || rows[i] >= N) return ORACLE_EINVAL;
  if (nrows == 0) return ORACLE_OK;
  int T = oracle_threads(nthreads, nrows);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * T);
  fwd_job* jobs = (fwd_job*)malloc(sizeof(fwd_job) * T);
  if (!th || !jobs) {
    free(th);
    free(jobs);
    return ORACLE_ENOMEM;
  }
  int rc = ORACLE_OK;
  for (int t = 0; t < T; ++t) {
    fwd_job J = {q, k, v, N, d, causal, scale, alibi, bmask, nb, dr, rows,
                 (int)((long)nrows * t / T), (int)((long)nrows * (t + 1) / T),
                 o, lse};
    jobs[t] = J;
    pthread_create(&th[t], NULL, fwd_worker, &jobs[t]);
  }
  for (int t = 0; t < T; ++t) {
    void* ret = NULL;
    pthread_join(th[t], &ret);
    if (ret) rc = ORACLE_ENOMEM;
  }
  free(th);
  free(jobs);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Backward                                                                   */
/* ------------------------------------------------------------------------ */
typedef struct {
  const double *q, *k, *v, *dO;
  int N, d, causal;
  double scale, alibi;
  const unsigned char* bmask;
  int nb;
  const dropout_spec* dr; /* NULL: no dropout */
  int r0, r1;          /* query rows [r0, r1) handled by this thread */
  const int* qpos;     /* qpos[r] = index of row r in the dQ output, or -1 */
  const int* kpos;     /* kpos[j] = index of key j in the dK/dV output, or -1 */
  int nkeys;
  double* dq;          /* shared; each row written by one thread only */
  double* Dvec;        /* shared [N] or NULL */
  double *dk, *dv;     /* private partial sums [nkeys][d] */
  int failed;
} bwd_job;

static void* bwd_worker(void* arg) {
  bwd_job* J = (bwd_job*)arg;
  const int N = J->N, d = J->d;
  double* p = (double*)malloc(sizeof(double) * (size_t)N);
  double* dp = (double*)malloc(sizeof(double) * (size_t)N);
  if (!p || !dp) {
    free(p);
    free(dp);
    J->failed = 1;
    return NULL;
  }
  for (int r = J->r0; r < J->r1; ++r) {
    int ncols;
    softmax_row(J->q, J->k, N, d, J->scale, J->alibi, J->causal, J->bmask, J->nb,
                r, p, &ncols);
    const double* dor = J->dO + (size_t)r * d;
    const double* qr = J->q + (size_t)r * d;
    /* dP_rj = <dO_r, v_j> (times Z_rj / q under dropout) and
     * D_r = sum_j P_rj dP_rj */
    double D = 0.0;
    for (int j = 0; j < ncols; ++j) {
      if (p[j] == 0.0) { /* removed (or underflowed) score: dS_rj = 0, no term */
        dp[j] = 0.0;
        continue;
      }
      const double* vj = J->v + (size_t)j * d;
      double s = 0.0;
      for (int c = 0; c < d; ++c) s += dor[c] * vj[c];
      if (J->dr) s = dropout_keep(J->dr, r, j) ? s * (256.0 / J->dr->t) : 0.0;
      dp[j] = s;
      D += p[j] * s;
    }
    if (J->Dvec) J->Dvec[r] = D;
    /* dS_rj = P_rj (dP_rj - D_r) */
    for (int j = 0; j < ncols; ++j) dp[j] = p[j] * (dp[j] - D);
    int qi = J->qpos[r];
    if (qi >= 0) {
      double* dqr = J->dq + (size_t)qi * d;
      for (int c = 0; c < d; ++c) dqr[c] = 0.0;
      for (int j = 0; j < ncols; ++j) {
        const double* kj = J->k + (size_t)j * d;
        for (int c = 0; c < d; ++c) dqr[c] += dp[j] * kj[c];
      }
      for (int c = 0; c < d; ++c) dqr[c] *= J->scale;
    }
    for (int j = 0; j < ncols; ++j) {
      int ki = J->kpos[j];
      if (ki < 0) continue;
      double* dkj = J->dk + (size_t)ki * d;
      double* dvj = J->dv + (size_t)ki * d;
      double ds = J->scale * dp[j];
      double pv = p[j]; /* the weight of dO_r in dV_j: Z_rj P_rj / q */
      if (J->dr) pv = dropout_keep(J->dr, r, j) ? pv * (256.0 / J->dr->t) : 0.0;
      for (int c = 0; c < d; ++c) {
        dkj[c] += ds * qr[c];
        dvj[c] += pv * dor[c];
      }
    }
  }
  free(p);
  free(dp);
  return NULL;
}

/* dQ[nrows][d] for the query rows in `rows`, dK/dV[nkeys][d] for the key rows
 * in `keys` (NULL lists: all N, in order; the count must then be N; a list
 * must not repeat an index), and
 * optionally D[N] (every row).  All N query rows always take part, because
 * every row contributes to dK and dV. */
int oracle_bwd(const double* q, const double* k, const double* v,
               const double* dO, int N, int d, double scale, double alibi,
               int causal, const unsigned char* bmask, int drop_t,
               unsigned long long seed, unsigned int offset, unsigned int head,
               const int* rows, int nrows, const int* keys, int nkeys,
               double* dq, double* dk, double* dv, double* Dvec, int nthreads) {
  if (!q || !k || !v || !dO || N < 1 || d < 1 || nrows < 0 || nkeys < 0)
    return ORACLE_EINVAL;
  if (drop_t < 1 || drop_t > 256) return ORACLE_EINVAL;
  dropout_spec drs = {drop_t, seed, offset, head};
  if ((!rows && nrows != N) || (!keys && nkeys != N)) return ORACLE_EINVAL;
  if ((nrows > 0 && !dq) || (nkeys > 0 && (!dk || !dv))) return ORACLE_EINVAL;
  int* qpos = (int*)malloc(sizeof(int) * (size_t)N);
  int* kpos = (int*)malloc(sizeof(int) * (size_t)N);
  if (!qpos || !kpos) {
    free(qpos);
    free(kpos);
    return ORACLE_ENOMEM;
  }
  for (int i = 0; i < N; ++i) qpos[i] = kpos[i] = -1;
  for (int i = 0; i < nrows; ++i) {
    int r = rows ? rows[i] : i;
    if (r < 0 || r >= N || qpos[r] >= 0) { /* out of range or repeated */
      free(qpos); free(kpos); return ORACLE_EINVAL;
    }
    qpos[r] = i;
  }
  for (int i = 0; i < nkeys; ++i) {
    int j = keys ? keys[i] : i;
    if (j < 0 || j >= N || kpos[j] >= 0) {
      free(qpos); free(kpos); return ORACLE_EINVAL;
    }
    kpos[j] = i;
  }
  int T = oracle_threads(nthreads, N);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * T);
  bwd_job* jobs = (bwd_job*)calloc((size_t)T, sizeof(bwd_job));
  size_t part = (size_t)nkeys * d;
  double* partial = (double*)calloc((size_t)T * 2 * (part ? part : 1), sizeof(double));
  if (!th || !jobs || !partial) {
    free(th); free(jobs); free(partial); free(qpos); free(kpos);
    return ORACLE_ENOMEM;
  }
  for (int t = 0; t < T; ++t) {
    bwd_job* J = &jobs[t];
    J->q = q; J->k = k; J->v = v; J->dO = dO;
    J->N = N; J->d = d; J->causal = causal; J->scale = scale; J->alibi = alibi;
    J->bmask = bmask; J->nb = (N + 127) / 128;
    J->dr = drop_t < 256 ? &drs : NULL;
    J->r0 = (int)((long)N * t / T);
    J->r1 = (int)((long)N * (t + 1) / T);
    J->qpos = qpos; J->kpos = kpos; J->nkeys = nkeys;
    J->dq = dq; J->Dvec = Dvec;
    J->dk = partial + (size_t)t * 2 * (part ? part : 1);
    J->dv = J->dk + part;
    pthread_create(&th[t], NULL, bwd_worker, J);
  }
  int rc = ORACLE_OK;
  for (int t = 0; t < T; ++t) {
    pthread_join(th[t], NULL);
    if (jobs[t].failed) rc = ORACLE_ENOMEM;
  }
  if (rc == ORACLE_OK && nkeys > 0) {
    memset(dk, 0, sizeof(double) * part);
    memset(dv, 0, sizeof(double) * part);
    for (int t = 0; t < T; ++t)
      for (size_t i = 0; i < part; ++i) {
        dk[i] += jobs[t].dk[i];
        dv[i] += jobs[t].dv[i];
      }
  }
  free(th); free(jobs); free(partial); free(qpos); free(kpos);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Blockwise (online) softmax forward, for the tiled == full invariant only.  */
/* Keys are visited in blocks X_j of `tile` columns.  Per page "突破单卡显存    */
/* 极限", section 2.1:                                                        */
/*   m = -inf, l = 0                                                          */
/*   per block: m_j = max(X_j); f_j = exp(X_j - m_j); l_j = sum(f_j)          */
/*              m_new = max(m, m_j)                                           */
/*              l_new = exp(m - m_new) l + exp(m_j - m_new) l_j               */
/*              f_j  <- f_j exp(m_j - m_new)                                  */
/* and, left implicit on the page: acc <- exp(m - m_new) acc + f_j V_j,       */
/* m <- m_new, l <- l_new.  At the end O = acc / l and LSE = m + log l.       */
/* ------------------------------------------------------------------------ */
typedef struct {
  const double *q, *k, *v;
  int N, d, causal, tile;
  double scale;
  int r0, r1;
  double *o, *lse;
  int failed;
} online_job;

static void* online_worker(void* arg) {
  online_job* J = (online_job*)arg;
  const int N = J->N, d = J->d, W = J->tile;
  double* x = (double*)malloc(sizeof(double) * (size_t)W);
  double* acc = (double*)malloc(sizeof(double) * (size_t)d);
  if (!x || !acc) {
    free(x);
    free(acc);
    J->failed = 1;
    return NULL;
  }
  for (int r = J->r0; r < J->r1; ++r) {
    const double* qr = J->q + (size_t)r * d;
    int ncols = J->causal ? r + 1 : N;
    double m = -INFINITY, l = 0.0;
    for (int c = 0; c < d; ++c) acc[c] = 0.0;
    for (int j0 = 0; j0 < ncols; j0 += W) {
      int w = ncols - j0 < W ? ncols - j0 : W;
      double mj = -INFINITY;
      for (int t = 0; t < w; ++t) {
        const double* kj = J->k + (size_t)(j0 + t) * d;
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += qr[c] * kj[c];
        x[t] = s * J->scale;
        if (x[t] > mj) mj = x[t];
      }
      double lj = 0.0;
      for (int t = 0; t < w; ++t) {
        x[t] = exp(x[t] - mj); /* f_j */
        lj += x[t];
      }
      double m_new = m > mj ? m : mj;
      double a_old = exp(m - m_new); /* 0 on the first block (m = -inf) */
      double a_blk = exp(mj - m_new);
      double l_new = a_old * l + a_blk * lj;
      for (int t = 0; t < w; ++t) x[t] *= a_blk; /* f_j rescale */
      for (int c = 0; c < d; ++c) acc[c] *= a_old;
      for (int t = 0; t < w; ++t) {
        const double* vj = J->v + (size_t)(j0 + t) * d;
        for (int c = 0; c < d; ++c) acc[c] += x[t] * vj[c];
      }
      m = m_new;
      l = l_new;
    }
    for (int c = 0; c < d; ++c) J->o[(size_t)r * d + c] = acc[c] / l;
    J->lse[r] = m + log(l);
  }
  free(x);
  free(acc);
  return NULL;
}

int oracle_online_fwd(const double* q, const double* k, const double* v, int N,
                      int d, double scale, int causal, int tile, double* o,
                      double* lse, int nthreads) {
  if (!q || !k || !v || !o || !lse || N < 1 || d < 1 || tile < 1)
    return ORACLE_EINVAL;
  int T = oracle_threads(nthreads, N);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * T);
  online_job* jobs = (online_job*)calloc((size_t)T, sizeof(online_job));
  if (!th || !jobs) {
    free(th);
    free(jobs);
    return ORACLE_ENOMEM;
  }
  for (int t = 0; t < T; ++t) {
    online_job* J = &jobs[t];
    J->q = q; J->k = k; J->v = v;
    J->N = N; J->d = d; J->causal = causal; J->tile = tile; J->scale = scale;
    J->r0 = (int)((long)N * t / T);
    J->r1 = (int)((long)N * (t + 1) / T);
    J->o = o; J->lse = lse;
    pthread_create(&th[t], NULL, online_worker, J);
  }
  int rc = ORACLE_OK;
  for (int t = 0; t < T; ++t) {
    pthread_join(th[t], NULL);
    if (jobs[t].failed) rc = ORACLE_ENOMEM;
  }
  free(th);
  free(jobs);
  return rc;
}

/* ------------------------------------------------------------------------ */
/* Decoding: Nq query rows (the last Nq positions) against Nk keys.          */
/* ------------------------------------------------------------------------ */
typedef struct {
  const double *q, *k, *v;
  int Nq, Nk, d, causal;
  double scale, alibi;
  int r0, r1;
  double *o, *lse;
} decode_job;

static void* decode_worker(void* arg) {
  decode_job* J = (decode_job*)arg;
  double* p = (double*)malloc(sizeof(double) * (size_t)J->Nk);
  if (!p) return (void*)1;
  for (int i = J->r0; i < J->r1; ++i) {
    /* keys 0 .. ncols-1 are visible to query row i */
    int ncols = J->causal ? J->Nk - J->Nq + i + 1 : J->Nk;
    const double* qi = J->q + (size_t)i * J->d;
    double m = -INFINITY;
    for (int j = 0; j < ncols; ++j) {
      const double* kj = J->k + (size_t)j * J->d;
      double s = 0.0;
      for (int c = 0; c < J->d; ++c) s += qi[c] * kj[c];
      s *= J->scale;
      s -= J->alibi * fabs((double)(J->Nk - J->Nq + i - j)); /* query at Nk-Nq+i */
      p[j] = s;
      if (s > m) m = s;
    }
    double z = 0.0;
    for (int j = 0; j < ncols; ++j) {
      p[j] = exp(p[j] - m);
      z += p[j];
    }
    double* orow = J->o + (size_t)i * J->d;
    for (int c = 0; c < J->d; ++c) orow[c] = 0.0;
    for (int j = 0; j < ncols; ++j) {
      const double* vj = J->v + (size_t)j * J->d;
      const double pj = p[j] / z;
      for (int c = 0; c < J->d; ++c) orow[c] += pj * vj[c];
    }
    if (J->lse) J->lse[i] = m + log(z);
  }
  free(p);
  return NULL;
}

/* O[Nq][d] and LSE[Nq] of Nq query rows q[Nq][d] against keys k[Nk][d] and
 * values v[Nk][d].  Causal needs Nq <= Nk (every row sees at least one key). */
int oracle_decode_fwd(const double* q, const double* k, const double* v, int Nq,
                      int Nk, int d, double scale, double alibi, int causal,
                      double* o, double* lse, int nthreads) {
  if (!q || !k || !v || !o || Nq < 1 || Nk < 1 || d < 1) return ORACLE_EINVAL;
  if (causal && Nq > Nk) return ORACLE_EINVAL;
  int T = oracle_threads(nthreads, Nq);
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * T);
  decode_job* jobs = (decode_job*)malloc(sizeof(decode_job) * T);
  if (!th || !jobs) {
    free(th);
    free(jobs);
    return ORACLE_ENOMEM;
  }
  int rc = ORACLE_OK;
  for (int t = 0; t < T; ++t) {
    decode_job J = {q, k, v, Nq, Nk, d, causal, scale, alibi,
                    (int)((long)Nq * t / T), (int)((long)Nq * (t + 1) / T), o, lse};
    jobs[t] = J;
    pthread_create(&th[t], NULL, decode_worker, &jobs[t]);
  }
  for (int t = 0; t < T; ++t) {
    void* ret = NULL;
    pthread_join(th[t], &ret);
    if (ret) rc = ORACLE_ENOMEM;
  }
  free(th);
  free(jobs);
  return rc;
}
