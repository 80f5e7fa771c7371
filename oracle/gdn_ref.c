/*
 * gdn_ref.c — fp64 CPU oracle for the gated delta rule (TEST INFRASTRUCTURE ONLY).
 *
 * Only tests, the smoke check and the benchmark's CPU-baseline leg may build, load or run
 * this file. It shares no code, header, table or helper with the CUDA library: it is the
 * plain definition of what the library computes, written out token by token in double
 * precision so a reader can check it against the definitions by eye.
 *
 * Definition followed (gated delta rule, Gated Delta Networks, Yang, Kautz & Hatamizadeh,
 * 2024; the "linear-attention scan" of sparkinfer v0.6.28 and the GDN layer of vllm.cpp
 * "vLLM, online serving"), per prompt n and value head h, key head hk = h / (H_v / H_k):
 *
 *     S   = initial state (or zero)                          d_v x d_k
 *     for each token t of the prompt, in order:
 *         q, k = q_t, k_t   (divided by sqrt(x.x + eps) when l2norm is on)
 *         g = exp(a_t)
 *         S = g S                                            decay
 *         delta = beta_t (v_t - S k)                         = -beta (g S_{t-1} k - v)
 *         S = S + delta k^T                                  rank-one write
 *         o_t = scale * S q                                  uses the updated state
 *         if t+1 is a requested checkpoint position: save S
 *     final state = S
 *
 * Checkpoint positions are prompt-relative token counts (the state after the first p
 * tokens of the segment); the per-prompt prefix-cache checkpoints of sparkinfer v0.6.28
 * (release notes, bullets 2-4) are snapshots of exactly this state.
 *
 * The only concurrency is across independent (prompt, value head) pairs; within a pair
 * every operation runs in the order written above.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
  int32_t num_seqs;
  const int32_t* cu_seqlens;   /* [N+1] */
  int32_t hk_heads, hv_heads, dk, dv;
  double scale;
  int32_t l2norm;
  double eps;
  const double *q, *k, *v, *a, *beta; /* [T][Hk][dk], [T][Hk][dk], [T][Hv][dv], [T][Hv] x2 */
  const double* init;                 /* [N][Hv][dv][dk] or NULL */
  const int32_t* ckpt_cu;             /* [N+1] or NULL */
  const int32_t* ckpt_pos;            /* [ckpt_cu[N]] */
  double* o;                          /* [T][Hv][dv] */
  double* ckpt;                       /* [ckpt_cu[N]][Hv][dv][dk] or NULL */
  double* final_state;                /* [N][Hv][dv][dk] */
  /* work distribution */
  int64_t next_unit;
  pthread_mutex_t lock;
} gdn_ref_job;

/* One (prompt n, value head h) pair, token by token. */
static void run_unit(const gdn_ref_job* J, int32_t n, int32_t h, double* S, double* qn,
                     double* kn) {
  const int32_t dk = J->dk, dv = J->dv, Hk = J->hk_heads, Hv = J->hv_heads;
  const int32_t hk = h / (Hv / Hk);
  const int32_t t0 = J->cu_seqlens[n], len = J->cu_seqlens[n + 1] - t0;
  const size_t state_elems = (size_t)dv * dk;

  if (J->init)
    memcpy(S, J->init + ((size_t)n * Hv + h) * state_elems, state_elems * sizeof(double));
  else
    memset(S, 0, state_elems * sizeof(double));

  int32_t c_next = 0, c_end = 0;
  if (J->ckpt_cu) {
    c_next = J->ckpt_cu[n];
    c_end = J->ckpt_cu[n + 1];
  }

  for (int32_t t = 0; t < len; ++t) {
    const size_t tok = (size_t)(t0 + t);
    const double* qt = J->q + (tok * Hk + hk) * dk;
    const double* kt = J->k + (tok * Hk + hk) * dk;
    const double* vt = J->v + (tok * Hv + h) * dv;
    const double g = exp(J->a[tok * Hv + h]);
    const double b = J->beta[tok * Hv + h];

    /* optional L2 normalisation of q and k */
    double qq = 0.0, kk = 0.0;
    for (int32_t j = 0; j < dk; ++j) {
      qq += qt[j] * qt[j];
      kk += kt[j] * kt[j];
    }
    const double qs = J->l2norm ? 1.0 / sqrt(qq + J->eps) : 1.0;
    const double ks = J->l2norm ? 1.0 / sqrt(kk + J->eps) : 1.0;
    for (int32_t j = 0; j < dk; ++j) {
      qn[j] = qt[j] * qs;
      kn[j] = kt[j] * ks;
    }

    double* ot = J->o + (tok * Hv + h) * dv;
    for (int32_t i = 0; i < dv; ++i) {
      double* Si = S + (size_t)i * dk;
      /* S = g S */
      for (int32_t j = 0; j < dk; ++j) Si[j] *= g;
      /* delta_i = beta (v_i - (S k)_i) */
      double sk = 0.0;
      for (int32_t j = 0; j < dk; ++j) sk += Si[j] * kn[j];
      const double delta = b * (vt[i] - sk);
      /* S_i += delta_i k^T */
      for (int32_t j = 0; j < dk; ++j) Si[j] += delta * kn[j];
      /* o_i = scale (S q)_i */
      double sq = 0.0;
      for (int32_t j = 0; j < dk; ++j) sq += Si[j] * qn[j];
      ot[i] = J->scale * sq;
    }

    while (c_next < c_end && J->ckpt_pos[c_next] == t + 1) {
      memcpy(J->ckpt + ((size_t)c_next * Hv + h) * state_elems, S,
             state_elems * sizeof(double));
      ++c_next;
    }
  }
  memcpy(J->final_state + ((size_t)n * Hv + h) * state_elems, S,
         state_elems * sizeof(double));
}

static void* worker(void* arg) {
  gdn_ref_job* J = (gdn_ref_job*)arg;
  const int64_t units = (int64_t)J->num_seqs * J->hv_heads;
  double* S = (double*)malloc(sizeof(double) * ((size_t)J->dv * J->dk + 2 * (size_t)J->dk));
  if (!S) return (void*)1;
  double* qn = S + (size_t)J->dv * J->dk;
  double* kn = qn + J->dk;
  for (;;) {
    pthread_mutex_lock(&J->lock);
    const int64_t u = J->next_unit++;
    pthread_mutex_unlock(&J->lock);
    if (u >= units) break;
    run_unit(J, (int32_t)(u / J->hv_heads), (int32_t)(u % J->hv_heads), S, qn, kn);
  }
  free(S);
  return NULL;
}

/* Returns 0 on success, -1 on invalid arguments, -2 when a thread could not start. */
int gdn_ref_prefill(int32_t num_seqs, const int32_t* cu_seqlens, int32_t hk_heads,
                    int32_t hv_heads, int32_t dk, int32_t dv, double scale, int32_t l2norm,
                    double eps, const double* q, const double* k, const double* v,
                    const double* a, const double* beta, const double* init,
                    const int32_t* ckpt_cu, const int32_t* ckpt_pos, double* o, double* ckpt,
                    double* final_state, int32_t num_threads) {
  if (num_seqs < 0 || hk_heads <= 0 || hv_heads <= 0 || hv_heads % hk_heads != 0 || dk <= 0 ||
      dv <= 0 || !cu_seqlens || !final_state)
    return -1;
  for (int32_t n = 0; n < num_seqs; ++n) {
    if (cu_seqlens[n + 1] < cu_seqlens[n]) return -1;
    if (ckpt_cu) {
      if (ckpt_cu[n + 1] < ckpt_cu[n]) return -1;
      const int32_t len = cu_seqlens[n + 1] - cu_seqlens[n];
      for (int32_t c = ckpt_cu[n]; c < ckpt_cu[n + 1]; ++c) {
        if (ckpt_pos[c] < 1 || ckpt_pos[c] > len) return -1;
        if (c > ckpt_cu[n] && ckpt_pos[c] <= ckpt_pos[c - 1]) return -1;
      }
    }
  }
  gdn_ref_job J;
  memset(&J, 0, sizeof(J));
  J.num_seqs = num_seqs;
  J.cu_seqlens = cu_seqlens;
  J.hk_heads = hk_heads;
  J.hv_heads = hv_heads;
  J.dk = dk;
  J.dv = dv;
  J.scale = scale;
  J.l2norm = l2norm;
  J.eps = eps;
  J.q = q;
  J.k = k;
  J.v = v;
  J.a = a;
  J.beta = beta;
  J.init = init;
  J.ckpt_cu = ckpt_cu;
  J.ckpt_pos = ckpt_pos;
  J.o = o;
  J.ckpt = ckpt;
  J.final_state = final_state;
  J.next_unit = 0;
  pthread_mutex_init(&J.lock, NULL);

  if (num_threads < 1) num_threads = 1;
  int rc = 0;
  if (num_threads == 1) {
    if (worker(&J) != NULL) rc = -2;
  } else {
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)num_threads);
    int started = 0;
    for (int i = 0; i < num_threads; ++i) {
      if (pthread_create(&th[i], NULL, worker, &J) != 0) break;
      ++started;
    }
    if (started == 0) rc = -2;
    for (int i = 0; i < started; ++i) {
      void* r = NULL;
      pthread_join(th[i], &r);
      if (r != NULL) rc = -2;
    }
    free(th);
  }
  pthread_mutex_destroy(&J.lock);
  return rc;
}

/* One decode token per sequence: the recurrence above applied once to S = states[slot[b]].
 * q, k: [B][Hk][dk]; v: [B][Hv][dv]; a, beta: [B][Hv]; states: [slots][Hv][dv][dk] updated
 * in place; o: [B][Hv][dv]. It is the prefill recurrence on a one-token prompt. */
int gdn_ref_decode(int32_t batch, int32_t hk_heads, int32_t hv_heads, int32_t dk, int32_t dv,
                   double scale, int32_t l2norm, double eps, const double* q, const double* k,
                   const double* v, const double* a, const double* beta, double* states,
                   const int32_t* slot, double* o) {
  if (batch < 0 || hk_heads <= 0 || hv_heads <= 0 || hv_heads % hk_heads != 0) return -1;
  const size_t state_elems = (size_t)dv * dk;
  double* qn = (double*)malloc(sizeof(double) * 2 * (size_t)dk);
  if (!qn) return -2;
  double* kn = qn + dk;
  for (int32_t b = 0; b < batch; ++b) {
    for (int32_t h = 0; h < hv_heads; ++h) {
      const int32_t hk = h / (hv_heads / hk_heads);
      const double* qt = q + ((size_t)b * hk_heads + hk) * dk;
      const double* kt = k + ((size_t)b * hk_heads + hk) * dk;
      const double* vt = v + ((size_t)b * hv_heads + h) * dv;
      const double g = exp(a[(size_t)b * hv_heads + h]);
      const double bb = beta[(size_t)b * hv_heads + h];
      double qq = 0.0, kk = 0.0;
      for (int32_t j = 0; j < dk; ++j) {
        qq += qt[j] * qt[j];
        kk += kt[j] * kt[j];
      }
      const double qs = l2norm ? 1.0 / sqrt(qq + eps) : 1.0;
      const double ks = l2norm ? 1.0 / sqrt(kk + eps) : 1.0;
      for (int32_t j = 0; j < dk; ++j) {
        qn[j] = qt[j] * qs;
        kn[j] = kt[j] * ks;
      }
      double* S = states + ((size_t)slot[b] * hv_heads + h) * state_elems;
      double* ot = o + ((size_t)b * hv_heads + h) * dv;
      for (int32_t i = 0; i < dv; ++i) {
        double* Si = S + (size_t)i * dk;
        for (int32_t j = 0; j < dk; ++j) Si[j] *= g;
        double sk = 0.0;
        for (int32_t j = 0; j < dk; ++j) sk += Si[j] * kn[j];
        const double delta = bb * (vt[i] - sk);
        for (int32_t j = 0; j < dk; ++j) Si[j] += delta * kn[j];
        double sq = 0.0;
        for (int32_t j = 0; j < dk; ++j) sq += Si[j] * qn[j];
        ot[i] = scale * sq;
      }
    }
  }
  free(qn);
  return 0;
}
