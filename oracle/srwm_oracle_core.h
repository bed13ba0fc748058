/*
 * srwm_oracle_core.h -- the body of the CPU oracle, written once and
 * instantiated twice by srwm_oracle.c: with REAL = double (the oracle proper)
 * and with REAL = float (used only to measure the fp32 rounding floor).
 *
 * TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may call this code.  The GPU library shares nothing with it.
 *
 * Before inclusion the includer defines:
 *   REAL      the arithmetic type
 *   EXP       the exponential for REAL (exp or expf)
 *   SFX(n)    a name suffixer (n##_f64 or n##_f32)
 *
 * Every step follows the SRWM definition of
 *   "Metalearning Continual Learning Algorithms", section 2.3,
 *   Eqs. (1)-(3) (single learning rate) and Eqs. (4)-(5) (four learning rates),
 * and the review "SRWM: letting a weight matrix learn to modify itself"
 * (of "A Modern Self-Referential Weight Matrix That Learns to Modify Itself"),
 * sections 2.2-2.4.  Notation: W has m = d_out + 2 d_in + n_lr rows and
 * d_in columns, d_in = d_out = d per head; its row blocks are, in order,
 * o (rows 0..d-1), k (d..2d-1), q (2d..3d-1) and beta (3d..m-1).
 */

/* phi: softmax over n entries.  The maximum is subtracted first; this leaves
 * the mathematical value unchanged and keeps exp() in range. */
static void SFX(softmax)(const REAL* in, REAL* out, int n)
{
    REAL mx = in[0];
    for (int i = 1; i < n; ++i)
        if (in[i] > mx) mx = in[i];
    REAL sum = 0;
    for (int i = 0; i < n; ++i) {
        out[i] = EXP(in[i] - mx);
        sum += out[i];
    }
    for (int i = 0; i < n; ++i) out[i] = out[i] / sum;
}

/* sigma: the logistic sigmoid. */
static REAL SFX(sigmoid)(REAL v) { return (REAL)1 / ((REAL)1 + EXP(-v)); }

/* out[r] = sum_c W[r,c] * vec[c]  (plain matrix-vector product, W row-major m x d). */
static void SFX(matvec)(const REAL* W, int m, int d, const REAL* vec, REAL* out)
{
    for (int r = 0; r < m; ++r) {
        REAL acc = 0;
        for (int c = 0; c < d; ++c) acc += W[(size_t)r * d + c] * vec[c];
        out[r] = acc;
    }
}

/*
 * The delta-rule self-update with given read/write addresses
 * (Eq. (2) and Eq. (3); per row block, Eqs. (4)-(5)):
 *   v    = W phi(q)            (read at the query address)
 *   vbar = W phi(k)            (read at the key address)
 *   W[r,:] += gate[r] * (v[r] - vbar[r]) * phi(k)
 * Both reads use the matrix before any write.  gate[r] is sigma(beta) of the
 * learning rate that governs row r.  scratch holds 2*m values.
 */
static void SFX(delta_update)(REAL* W, int m, int d, const REAL* phi_k, const REAL* phi_q,
                              const REAL* gate, REAL* scratch)
{
    REAL* v = scratch;
    REAL* vbar = scratch + m;
    SFX(matvec)(W, m, d, phi_q, v);
    SFX(matvec)(W, m, d, phi_k, vbar);
    for (int r = 0; r < m; ++r) {
        const REAL coef = gate[r] * (v[r] - vbar[r]);
        for (int c = 0; c < d; ++c) W[(size_t)r * d + c] += coef * phi_k[c];
    }
}

/*
 * One (sequence, head) stream: T steps of Eqs. (1)-(3) / (4)-(5).
 *   x      : the stream's inputs, step t at x + t*x_stride (d floats each)
 *   W      : m x d state, holds W_0 on entry and W_T on exit
 *   y      : step t's output at y + t*y_stride (d values each)
 *   work   : 6*m + 3*d values of scratch
 */
static void SFX(run_stream)(const float* x, size_t x_stride, REAL* W, int T, int d, int n_lr,
                            int softmax_input, REAL* y, size_t y_stride, REAL* work)
{
    const int m = 3 * d + n_lr;
    REAL* u     = work;           /* d: the input u_t (after phi when softmax_input) */
    REAL* z     = u + d;          /* m: [o_t, k_t, q_t, beta_t] = W_{t-1} u_t          */
    REAL* phi_k = z + m;          /* d */
    REAL* phi_q = phi_k + d;      /* d */
    REAL* gate  = phi_q + d;      /* m: sigma(beta) of the block that owns each row   */
    REAL* scr   = gate + m;       /* 2m: v and vbar for delta_update                  */

    for (int t = 0; t < T; ++t) {
        const float* xt = x + (size_t)t * x_stride;
        /* The input, with or without phi (section 2.3: supervised settings use
         * none, the RL setting applies softmax). */
        for (int c = 0; c < d; ++c) u[c] = (REAL)xt[c];
        if (softmax_input) SFX(softmax)(u, u, d);

        /* Eq. (1): [o_t, k_t, q_t, beta_t] = W_{t-1} u_t. */
        SFX(matvec)(W, m, d, u, z);

        /* The output comes from the pre-update matrix W_{t-1}. */
        REAL* yt = y + (size_t)t * y_stride;
        for (int c = 0; c < d; ++c) yt[c] = z[c];

        /* phi(k_t), phi(q_t). */
        SFX(softmax)(z + d, phi_k, d);
        SFX(softmax)(z + 2 * d, phi_q, d);

        /* Learning rates: one sigma(beta_t) for every row (Eq. (3)), or one per
         * row block o/k/q/beta with beta_t = [b^o, b^k, b^q, b^b] (Eq. (5)). */
        for (int r = 0; r < m; ++r) {
            int blk = 0;
            if (n_lr == 4) blk = (r < 3 * d) ? r / d : 3;
            gate[r] = SFX(sigmoid)(z[3 * d + blk]);
        }

        /* Eqs. (2)-(3): W_t = W_{t-1} + sigma(beta)(v_t - vbar_t) (x) phi(k_t). */
        SFX(delta_update)(W, m, d, phi_k, phi_q, gate, scr);
    }
}

typedef struct {
    const float* x;
    const float* W_init;
    int W_init_per_sequence;
    int B, T, H, d, n_lr, softmax_input;
    REAL* y;
    REAL* W_final;
    long long first_pair, end_pair;
    int failed;
} SFX(job_t);

static void* SFX(job_main)(void* arg)
{
    SFX(job_t)* job = (SFX(job_t)*)arg;
    const int d = job->d, H = job->H, T = job->T;
    const int m = 3 * d + job->n_lr;
    const size_t md = (size_t)m * d;
    REAL* work = (REAL*)malloc(sizeof(REAL) * (size_t)(6 * m + 3 * d));
    if (!work) { job->failed = 1; return NULL; }
    for (long long p = job->first_pair; p < job->end_pair; ++p) {
        const int b = (int)(p / H), h = (int)(p % H);
        /* W_0 is shared by every sequence; each sequence evolves its own copy. */
        const float* w0 = job->W_init_per_sequence ? job->W_init + (size_t)p * md
                                                   : job->W_init + (size_t)h * md;
        REAL* W = job->W_final + (size_t)p * md;
        for (size_t i = 0; i < md; ++i) W[i] = (REAL)w0[i];
        /* Layout [B, T, H, d]: head h owns coordinates h*d .. h*d+d-1 of the
         * D = H*d wide input at every step. */
        const float* xs = job->x + ((size_t)b * T * H + h) * d;
        REAL* ys = job->y + ((size_t)b * T * H + h) * d;
        SFX(run_stream)(xs, (size_t)H * d, W, T, d, job->n_lr, job->softmax_input, ys,
                        (size_t)H * d, work);
    }
    free(work);
    return NULL;
}

static int SFX(forward)(const float* x, const float* W_init, int W_init_per_sequence, int B,
                        int T, int H, int d, int n_lr, int softmax_input, REAL* y,
                        REAL* W_final, int n_threads)
{
    if (!W_init || !W_final || (T > 0 && (!x || !y))) return 1;
    if (B <= 0 || H <= 0 || d <= 0 || T < 0) return 2;
    if (n_lr != 1 && n_lr != 4) return 3;
    const long long pairs = (long long)B * H;
    if (n_threads < 1) n_threads = 1;
    if (n_threads > pairs) n_threads = (int)pairs;
    SFX(job_t)* jobs = (SFX(job_t)*)calloc((size_t)n_threads, sizeof(SFX(job_t)));
    pthread_t* tids = (pthread_t*)calloc((size_t)n_threads, sizeof(pthread_t));
    if (!jobs || !tids) { free(jobs); free(tids); return 4; }
    for (int i = 0; i < n_threads; ++i) {
        SFX(job_t)* j = &jobs[i];
        j->x = x; j->W_init = W_init; j->W_init_per_sequence = W_init_per_sequence;
        j->B = B; j->T = T; j->H = H; j->d = d; j->n_lr = n_lr;
        j->softmax_input = softmax_input; j->y = y; j->W_final = W_final;
        j->first_pair = pairs * i / n_threads;
        j->end_pair = pairs * (i + 1) / n_threads;
    }
    int rc = 0;
    if (n_threads == 1) {
        SFX(job_main)(&jobs[0]);
    } else {
        int started = 0;
        for (int i = 0; i < n_threads; ++i) {
            if (pthread_create(&tids[i], NULL, SFX(job_main), &jobs[i]) != 0) break;
            ++started;
        }
        for (int i = 0; i < started; ++i) pthread_join(tids[i], NULL);
        for (int i = started; i < n_threads; ++i) SFX(job_main)(&jobs[i]);
    }
    for (int i = 0; i < n_threads; ++i) rc |= jobs[i].failed ? 4 : 0;
    free(jobs);
    free(tids);
    return rc;
}
