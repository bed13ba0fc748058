/*
 * srwm_oracle.c -- plain, slow, obviously correct CPU oracle of the
 * Self-Referential Weight Matrix (SRWM) forward recurrence.
 *
 * TEST INFRASTRUCTURE.  Only tests/, __graft_entry__.smoke() and the
 * benchmark's cpu_baseline / reference leg may load or run this library.  It
 * shares no code, header, table or helper with the CUDA library; the two meet
 * only through the seeded input generator, which holds none of the method's
 * arithmetic.
 *
 * What it computes, per (sequence b, head h) stream, is the SRWM of
 * "Metalearning Continual Learning Algorithms", section 2.3:
 *   Eq. (1)  [o_t, k_t, q_t, beta_t] = W_{t-1} u_t
 *   Eq. (2)  v_t = W_{t-1} phi(q_t),  vbar_t = W_{t-1} phi(k_t)
 *   Eq. (3)  W_t = W_{t-1} + sigma(beta_t) (v_t - vbar_t) (x) phi(k_t)
 * and its four-learning-rate version, Eqs. (4)-(5), where each row block
 * o/k/q/beta takes its own sigma(beta_t^X).  The output y_t = o_t is read from
 * the pre-update matrix (review of "A Modern Self-Referential Weight Matrix
 * That Learns to Modify Itself", section 2.2, on time ordering).  Heads are
 * independent (same review, section 2.4); W_0 is shared by every sequence.
 *
 * Each stream is a plain loop over t with plain nested loops inside; the only
 * parallelism is over independent (b, h) streams (pthreads), which reorders no
 * arithmetic inside a stream.
 *
 * Readings where the pages leave a step open:
 *   - row-block order [o; k; q; beta], beta_t = [b^o, b^k, b^q, b^b];
 *   - rows of block X use sigma(b^X); the four beta rows use sigma(b^b);
 *   - every read in a step uses W_{t-1}; all blocks update at once;
 *   - softmax subtracts the maximum first (value-identical);
 *   - with softmax_input, phi acts on each head's own d inputs.
 */
#include <math.h>
#include <pthread.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>

#define REAL double
#define EXP exp
#define SFX(n) n##_f64
#include "srwm_oracle_core.h"
#undef REAL
#undef EXP
#undef SFX

#define REAL float
#define EXP expf
#define SFX(n) n##_f32
#include "srwm_oracle_core.h"
#undef REAL
#undef EXP
#undef SFX

/*
 * Forward recurrence in double precision from fp32 inputs.
 *   x       [B, T, H, d] fp32 (may be NULL when T == 0)
 *   W_init  [H, m, d] fp32 shared by all sequences (W_init_per_sequence == 0)
 *           or [B, H, m, d] fp32, one state per sequence (== 1)
 *   y       [B, T, H, d] double
 *   W_final [B, H, m, d] double
 * Returns 0 on success, 1 null pointer, 2 bad shape, 3 unsupported n_lr,
 * 4 out of host memory.
 */
int srwm_oracle_forward_f64(const float* x, const float* W_init, int W_init_per_sequence, int B,
                            int T, int H, int d, int n_lr, int softmax_input, double* y,
                            double* W_final, int n_threads)
{
    return forward_f64(x, W_init, W_init_per_sequence, B, T, H, d, n_lr, softmax_input, y,
                       W_final, n_threads);
}

/* The same recurrence, same operation order, in float: it measures how far
 * plain fp32 arithmetic drifts from the double result (the fp32 floor). */
int srwm_oracle_forward_f32(const float* x, const float* W_init, int W_init_per_sequence, int B,
                            int T, int H, int d, int n_lr, int softmax_input, float* y,
                            float* W_final, int n_threads)
{
    return forward_f32(x, W_init, W_init_per_sequence, B, T, H, d, n_lr, softmax_input, y,
                       W_final, n_threads);
}

/*
 * One delta-rule self-update with the addresses given instead of generated
 * (Eqs. (2)-(3); per block, Eq. (5)):  W[r,:] += gate[r] (W phi_q - W phi_k)[r] phi_k.
 * W is m x d row-major double, updated in place.  Returns 0, or 1 / 2 / 4 as above.
 */
int srwm_oracle_delta_update(double* W, int m, int d, const double* phi_k, const double* phi_q,
                             const double* gate_of_row)
{
    if (!W || !phi_k || !phi_q || !gate_of_row) return 1;
    if (m <= 0 || d <= 0) return 2;
    double* scratch = (double*)malloc(sizeof(double) * 2 * (size_t)m);
    if (!scratch) return 4;
    delta_update_f64(W, m, d, phi_k, phi_q, gate_of_row, scratch);
    free(scratch);
    return 0;
}
