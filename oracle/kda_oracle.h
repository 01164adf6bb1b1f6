/*
 * kda_oracle.h -- interface of the fp64 CPU oracle (test infrastructure only).
 *
 * The oracle is independent of the CUDA library: it includes none of its headers and
 * the library includes none of these.  Layouts mirror the library's so that the same
 * seeded tensors can be handed to both:
 *   q, k, v : [T_tot, H, d]   bf16 bit patterns (qkv_is_f32 = 0) or float32 (= 1)
 *   g       : [T_tot, H, d]   float32, natural-log per-channel decay (alpha = exp(g))
 *   beta    : [T_tot, H]      float32
 *   S_in    : [N, H, d, d]    float32 or NULL (zeros); row = d_k channel, column = d_v
 *   cu_seqlens [N+1], ckpt_off [N+1] / ckpt_pos [] : packed-sequence and checkpoint CSR
 */
#ifndef KDA_ORACLE_H
#define KDA_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { KDA_REF_OK = 0, KDA_REF_ERR_ARG = 1, KDA_REF_ERR_ALLOC = 2 };

typedef struct {
  const void* q;
  const void* k;
  const void* v;
  int qkv_is_f32;
  const float* g;
  const float* beta;
  const float* S_in;          /* may be NULL */
  const int32_t* cu_seqlens;  /* [n_seq + 1] */
  int n_seq, H, d;
  const int32_t* ckpt_off;    /* [n_seq + 1] or NULL */
  const int32_t* ckpt_pos;    /* positions in (0, len], strictly increasing per sequence */
  const int64_t* units;       /* (seq * H + head) to compute, or NULL for all */
  int64_t n_units;
  double* o;                  /* [T_tot, H, d], or [n_o_rows, H, d] when o_rows != NULL; may be NULL */
  const int64_t* o_rows;      /* ascending packed rows whose outputs are kept, or NULL */
  int64_t n_o_rows;
  double* S_out;              /* [N, H, d, d] or NULL */
  double* ckpts;              /* [n_ckpt_total, H, d, d] or NULL */
  int n_threads;              /* <= 0: one per online CPU */
} kda_ref_args;

/* Runs the per-token recurrence for every requested unit; returns KDA_REF_OK or an
 * error code.  *threads_used (if non-NULL) receives the worker-thread count. */
int kda_ref_run(const kda_ref_args* args, int* threads_used);

#ifdef __cplusplus
}
#endif

#endif
