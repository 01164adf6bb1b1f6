/*
 * kda_oracle.c -- fp64 CPU oracle for the Kimi Delta Attention (KDA) recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or calls this
 * file; only the test-suite, the smoke check and the benchmark's CPU-baseline leg do.
 * It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition, applied token by token in fp64):
 *
 *   "Kimi K3.1 Pro 架构完全拆解", section 3.1 (single-head recurrence):
 *       S_t = (I - beta_t k_t k_t^T) Diag(alpha_t) S_{t-1} + beta_t k_t v_t^T
 *       o_t = S_t^T q_t,           alpha_t = exp(g_t) per d_k channel (section 3.2,
 *                                  bounded log-decay g in (g_min, 0), natural log)
 *
 *   The product (I - beta k k^T) X is evaluated with the associativity
 *   X - beta k (k^T X), which is the delta-rule form printed in
 *   "Kimi K3 ... 服務性能" (SemiAnalysis translation), section 6 "FlashKDA 演算法":
 *       X = Diag(alpha_t) S_{t-1};  u_t = beta_t (v_t - X^T k_t);
 *       S_t = X + k_t u_t^T;        o_t = S_t^T q_t.
 *   No blocking, no chunking, no reordering beyond that identity.
 *
 * S is d_k x d_v, row index = d_k channel (the channel alpha scales), column = d_v.
 * Inputs are widened exactly to fp64 (bf16 -> fp32 -> fp64 are exact conversions).
 *
 * Checkpoints ("部署 Kimi K3 ...", section 3.2: the kernel persists the state at
 * hash-aligned positions): position p of sequence i is the number of that sequence's
 * tokens consumed in this call; the snapshot is S after its p-th token.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include "kda_oracle.h"

static double widen_bf16(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double load_elem(const void* base, int is_f32, int64_t idx) {
  if (is_f32) return (double)((const float*)base)[idx];
  return widen_bf16(((const uint16_t*)base)[idx]);
}

typedef struct {
  const kda_ref_args* a;
  int64_t next_unit; /* shared work counter (atomic) */
  int status;
} pool_t;

/* Map a packed token row to its slot in o: all rows, or the listed rows only. */
static int64_t o_slot(const kda_ref_args* a, int64_t row) {
  if (a->o_rows == NULL) return row;
  int64_t lo = 0, hi = a->n_o_rows - 1;
  while (lo <= hi) {
    int64_t mid = lo + (hi - lo) / 2;
    if (a->o_rows[mid] == row) return mid;
    if (a->o_rows[mid] < row) lo = mid + 1; else hi = mid - 1;
  }
  return -1;
}

/* One (sequence, head) unit: the literal per-token recurrence in fp64. */
static int run_unit(const kda_ref_args* a, int seq, int h, double* S, double* x, double* w) {
  const int H = a->H, d = a->d;
  const int64_t bos = a->cu_seqlens[seq];
  const int64_t len = (int64_t)a->cu_seqlens[seq + 1] - bos;
  const int64_t dd = (int64_t)d * d;

  /* S_0: the caller's initial state, or zeros. */
  if (a->S_in) {
    const float* s0 = a->S_in + ((int64_t)seq * H + h) * dd;
    for (int64_t e = 0; e < dd; ++e) S[e] = (double)s0[e];
  } else {
    memset(S, 0, sizeof(double) * (size_t)dd);
  }

  int c_begin = 0, c_end = 0, c = 0;
  if (a->ckpt_off) { c_begin = a->ckpt_off[seq]; c_end = a->ckpt_off[seq + 1]; c = c_begin; }

  double* q = x;          /* d */
  double* k = x + d;      /* d */
  double* v = x + 2 * d;  /* d */
  double* al = x + 3 * d; /* d: alpha = exp(g) */
  double* u = w;          /* d */

  for (int64_t t = 0; t < len; ++t) {
    const int64_t row = bos + t;
    const int64_t base = (row * H + h) * (int64_t)d;
    for (int i = 0; i < d; ++i) {
      q[i] = load_elem(a->q, a->qkv_is_f32, base + i);
      k[i] = load_elem(a->k, a->qkv_is_f32, base + i);
      v[i] = load_elem(a->v, a->qkv_is_f32, base + i);
      al[i] = exp((double)a->g[base + i]);
    }
    const double beta = (double)a->beta[row * H + h];

    /* X = Diag(alpha) S : scale row i (the d_k channel) by alpha_i. */
    for (int i = 0; i < d; ++i) {
      double* Si = S + (int64_t)i * d;
      for (int j = 0; j < d; ++j) Si[j] *= al[i];
    }
    /* u = beta (v - X^T k) */
    for (int j = 0; j < d; ++j) u[j] = 0.0;
    for (int i = 0; i < d; ++i) {
      const double* Si = S + (int64_t)i * d;
      for (int j = 0; j < d; ++j) u[j] += Si[j] * k[i];
    }
    for (int j = 0; j < d; ++j) u[j] = beta * (v[j] - u[j]);
    /* S = X + k u^T */
    for (int i = 0; i < d; ++i) {
      double* Si = S + (int64_t)i * d;
      for (int j = 0; j < d; ++j) Si[j] += k[i] * u[j];
    }
    /* o = S^T q */
    if (a->o) {
      int64_t slot = o_slot(a, row);
      if (slot >= 0) {
        double* o = a->o + (slot * H + h) * (int64_t)d;
        for (int j = 0; j < d; ++j) o[j] = 0.0;
        for (int i = 0; i < d; ++i) {
          const double* Si = S + (int64_t)i * d;
          for (int j = 0; j < d; ++j) o[j] += Si[j] * q[i];
        }
      }
    }
    /* checkpoint after the (t+1)-th token of this sequence */
    if (c < c_end && a->ckpt_pos[c] == t + 1) {
      if (a->ckpts) memcpy(a->ckpts + ((int64_t)c * H + h) * dd, S, sizeof(double) * (size_t)dd);
      ++c;
    }
  }
  if (c != c_end) return KDA_REF_ERR_ARG; /* a requested position was never reached */
  if (a->S_out) memcpy(a->S_out + ((int64_t)seq * H + h) * dd, S, sizeof(double) * (size_t)dd);
  return KDA_REF_OK;
}

static void* worker(void* p) {
  pool_t* pool = (pool_t*)p;
  const kda_ref_args* a = pool->a;
  const int d = a->d;
  double* S = (double*)malloc(sizeof(double) * (size_t)d * d);
  double* x = (double*)malloc(sizeof(double) * 4 * (size_t)d);
  double* w = (double*)malloc(sizeof(double) * (size_t)d);
  if (!S || !x || !w) {
    __atomic_store_n(&pool->status, KDA_REF_ERR_ALLOC, __ATOMIC_RELAXED);
    free(S); free(x); free(w);
    return NULL;
  }
  const int64_t total = a->units ? a->n_units : (int64_t)a->n_seq * a->H;
  for (;;) {
    int64_t idx = __atomic_fetch_add(&pool->next_unit, 1, __ATOMIC_RELAXED);
    if (idx >= total) break;
    int64_t unit = a->units ? a->units[idx] : idx;
    int st = run_unit(a, (int)(unit / a->H), (int)(unit % a->H), S, x, w);
    if (st != KDA_REF_OK) __atomic_store_n(&pool->status, st, __ATOMIC_RELAXED);
  }
  free(S); free(x); free(w);
  return NULL;
}

static int validate(const kda_ref_args* a) {
  if (!a || !a->q || !a->k || !a->v || !a->g || !a->beta || !a->cu_seqlens) return KDA_REF_ERR_ARG;
  if (a->n_seq < 0 || a->H <= 0 || a->d <= 0) return KDA_REF_ERR_ARG;
  if (a->cu_seqlens[0] != 0) return KDA_REF_ERR_ARG;
  for (int s = 0; s < a->n_seq; ++s) {
    if (a->cu_seqlens[s + 1] < a->cu_seqlens[s]) return KDA_REF_ERR_ARG;
    if (a->ckpt_off) {
      if (!a->ckpt_pos || a->ckpt_off[s + 1] < a->ckpt_off[s]) return KDA_REF_ERR_ARG;
      int32_t len = a->cu_seqlens[s + 1] - a->cu_seqlens[s];
      int32_t prev = 0;
      for (int c = a->ckpt_off[s]; c < a->ckpt_off[s + 1]; ++c) {
        if (a->ckpt_pos[c] <= prev || a->ckpt_pos[c] > len) return KDA_REF_ERR_ARG;
        prev = a->ckpt_pos[c];
      }
    }
  }
  if (a->ckpt_off && a->ckpt_off[0] != 0) return KDA_REF_ERR_ARG;
  if (a->units) {
    for (int64_t u = 0; u < a->n_units; ++u)
      if (a->units[u] < 0 || a->units[u] >= (int64_t)a->n_seq * a->H) return KDA_REF_ERR_ARG;
  }
  if (a->o_rows) {
    for (int64_t r = 1; r < a->n_o_rows; ++r)
      if (a->o_rows[r] <= a->o_rows[r - 1]) return KDA_REF_ERR_ARG;
  }
  return KDA_REF_OK;
}

int kda_ref_run(const kda_ref_args* a, int* threads_used) {
  int st = validate(a);
  if (st != KDA_REF_OK) return st;
  const int64_t total = a->units ? a->n_units : (int64_t)a->n_seq * a->H;
  long nt = a->n_threads > 0 ? a->n_threads : sysconf(_SC_NPROCESSORS_ONLN);
  if (nt < 1) nt = 1;
  if (nt > total) nt = total > 0 ? (long)total : 1;
  if (nt > 1024) nt = 1024;
  if (threads_used) *threads_used = (int)nt;

  pool_t pool;
  pool.a = a;
  pool.next_unit = 0;
  pool.status = KDA_REF_OK;
  if (nt == 1) {
    worker(&pool);
    return pool.status;
  }
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nt);
  if (!th) return KDA_REF_ERR_ALLOC;
  long started = 0;
  for (; started < nt; ++started)
    if (pthread_create(&th[started], NULL, worker, &pool) != 0) break;
  if (started == 0) worker(&pool);
  for (long i = 0; i < started; ++i) pthread_join(th[i], NULL);
  free(th);
  return pool.status;
}
