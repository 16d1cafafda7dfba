/*
 * fp64 CPU oracle for the Mamba-2 SSD forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path calls,
 * links or loads this file; only the tests, the smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code with the CUDA path.
 *
 * Everything is computed in double precision from the exact (widened) input
 * values.  Functions, and the passage each follows:
 *
 *   oracle_ssd_recurrence  the selective-SSM recurrence of "State Space Duality
 *                          and Mamba-2" (section "The Mathematical Bridge") with
 *                          the scalar-identity transition A_t = a_t I, written
 *                          per head:  h_t = exp(dt_t A_h) h_{t-1} + dt_t x_t B_t^T,
 *                          y_t = h_t C_t + D_h x_t.  Packed documents reset the
 *                          state at each document start ("Parallel Scan and
 *                          Hardware-Aware SSM Kernels", "When it breaks",
 *                          variable-length batching).
 *   oracle_ssd_quadratic   the same operator as one lower-triangular matrix
 *                          M = (C B^T) o L, L_ij = prod_{k=j+1..i} a_k
 *                          ("State Space Duality and Mamba-2", the 1-SS matrix
 *                          entry and the Hadamard factorisation), plus the
 *                          initial-state term.  O(L^2): tiny inputs only.
 *   oracle_ssd_chunked     the SSD block decomposition ("The SSD Block
 *                          Decomposition Algorithm": diagonal blocks, chunk
 *                          state summaries, inter-chunk state passing, chunk
 *                          state projection), with chunk states composed over
 *                          splits by the affine-step composition rule
 *                          ("Parallel Scan ...", "The scan").
 *   oracle_ssd_backward    gradients of the recurrence's outputs (y and the
 *                          final state) with respect to every input, by reverse-
 *                          mode differentiation of the recurrence itself, taken
 *                          backwards in time from the stored per-token states
 *                          (the states the backward pass needs, "Parallel Scan and
 *                          Hardware-Aware SSM Kernels", "Why the kernel matters
 *                          more than the algorithm"), batch rows or packed
 *                          documents.
 *   oracle_segsum          seg(i, j) = sum_{k=j+1..i} l_k for j <= i, -inf
 *                          above the diagonal, accumulated from the diagonal
 *                          leftwards (no prefix subtraction).
 *   oracle_diff_segsum_f32 the prefix-subtraction ("diff segsum") comparator of
 *                          "GPU Hierarchy Meets Structured Matrices": an fp32
 *                          inclusive cumsum in Kogge-Stone (log-step) order,
 *                          then cum_i - cum_j.  It is the known-unstable form
 *                          the stability tests must show failing.
 *
 * Conventions shared by the SSD functions:
 *   x (batch, L, H, P)   dt (batch, L, H)   A (H)   D (H) or NULL
 *   B, C (batch, L, G, N); head h uses group h / (H / G)
 *   state per (row-or-document, head) is a (P, N) matrix
 *   init / final (nst, H, P, N), nst = batch, or ndocs when cu_seqlens != NULL
 *   cu_seqlens (ndocs + 1) or NULL; when given, batch == 1 and every document
 *   starts from its own initial state (or zero).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX_X(b, t, h, p) ((((int64_t)(b) * L + (t)) * H + (h)) * P + (p))
#define IDX_DT(b, t, h) (((int64_t)(b) * L + (t)) * H + (h))
#define IDX_BC(b, t, g, n) ((((int64_t)(b) * L + (t)) * G + (g)) * N + (n))
#define IDX_S(s, h, p, n) ((((int64_t)(s) * H + (h)) * P + (p)) * N + (n))

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* document index of every token of row 0 (varlen), or -1 for plain batches */
static int doc_of(const int32_t* cu, int ndocs, int64_t t) {
    int lo = 0, hi = ndocs - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) / 2;
        if (cu[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* ---------------------------------------------------------------------- */
/* Sequential recurrence                                                   */
/* ---------------------------------------------------------------------- */
void oracle_ssd_recurrence(int64_t batch, int64_t L, int H, int P, int N, int G,
                           const double* x, const double* dt, const double* A,
                           const double* B, const double* C, const double* D,
                           const double* init, const int32_t* cu, int ndocs,
                           double* y, double* final_states, int nthreads) {
    const int hpg = H / G;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t b = 0; b < batch; ++b) {
        for (int h = 0; h < H; ++h) {
            const int g = h / hpg;
            double* S = (double*)malloc(sizeof(double) * (size_t)P * N);
            int doc = 0;
            for (int64_t t = 0; t < L; ++t) {
                /* (re)start: the sequence start, or a document start */
                int start = (t == 0);
                if (cu && t > 0 && doc + 1 < ndocs && t == cu[doc + 1]) { ++doc; start = 1; }
                if (start) {
                    const int s = cu ? doc : (int)b;
                    for (int p = 0; p < P; ++p)
                        for (int n = 0; n < N; ++n)
                            S[p * N + n] = init ? init[IDX_S(s, h, p, n)] : 0.0;
                }
                const double d = dt[IDX_DT(b, t, h)];
                const double a = exp(d * A[h]);
                for (int p = 0; p < P; ++p) {
                    const double u = d * x[IDX_X(b, t, h, p)];
                    double acc = 0.0;
                    for (int n = 0; n < N; ++n) {
                        double v = a * S[p * N + n] + u * B[IDX_BC(b, t, g, n)];
                        S[p * N + n] = v;
                        acc += v * C[IDX_BC(b, t, g, n)];
                    }
                    y[IDX_X(b, t, h, p)] = acc + (D ? D[h] * x[IDX_X(b, t, h, p)] : 0.0);
                }
                /* end of the sequence or of a document: record its state */
                int end = (t == L - 1) || (cu && doc + 1 < ndocs && t + 1 == cu[doc + 1]);
                if (end && final_states) {
                    const int s = cu ? doc : (int)b;
                    for (int p = 0; p < P; ++p)
                        for (int n = 0; n < N; ++n)
                            final_states[IDX_S(s, h, p, n)] = S[p * N + n];
                }
            }
            free(S);
        }
    }
}

/* ---------------------------------------------------------------------- */
/* Backward pass of the recurrence (reverse mode, backwards in time)        */
/* ---------------------------------------------------------------------- */
/* With S_t = a_t S_{t-1} + dt_t x_t B_t^T, a_t = exp(dt_t A_h), and
 * y_t = S_t C_t + D_h x_t, the adjoint Lam_t of S_t (the gradient of the loss
 * <dy, y> + <dfin, S_final> with respect to S_t, all later uses included) obeys
 *   Lam_t = dy_t C_t^T + a_{t+1} Lam_{t+1},  Lam_e = dfin + dy_e C_e^T at an end e
 * and each token's inputs collect
 *   dx_t  = dt_t Lam_t B_t + D_h dy_t
 *   dB_t += dt_t Lam_t^T x_t              (summed over the heads of the group)
 *   dC_t += S_t^T dy_t                    (summed over the heads of the group)
 *   dl_t  = a_t <Lam_t, S_{t-1}>          (the log-decay l_t = dt_t A_h)
 *   ddt_t = x_t . (Lam_t B_t) + A_h dl_t
 *   dA_h += dt_t dl_t,  dD_h += dy_t . x_t
 * and a start's initial state gets a_s Lam_s.  With packed documents
 * (cu != NULL, batch 1) every document is its own sequence: its state starts
 * from init[d] (or zero), its final state is dfin[d]'s, and no adjoint crosses
 * a document boundary.
 * Outputs are written (not accumulated into): dx (batch, L, H, P),
 * ddt (batch, L, H), dA (H), dB, dC (batch, L, G, N), dD (H) or NULL,
 * dinit (nst, H, P, N) or NULL; nst = ndocs with cu, else batch.  dfin may be
 * NULL (zero). */
void oracle_ssd_backward(int64_t batch, int64_t L, int H, int P, int N, int G,
                         const double* x, const double* dt, const double* A,
                         const double* B, const double* C, const double* D,
                         const double* init, const int32_t* cu, int ndocs,
                         const double* dy, const double* dfin,
                         double* dx, double* ddt, double* dA, double* dB, double* dC,
                         double* dD, double* dinit, int nthreads) {
    const int hpg = H / G;
    double* dA_part = (double*)calloc((size_t)batch * H, sizeof(double));
    double* dD_part = (double*)calloc((size_t)batch * H, sizeof(double));
    memset(dB, 0, sizeof(double) * (size_t)batch * L * G * N);
    memset(dC, 0, sizeof(double) * (size_t)batch * L * G * N);
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for collapse(2) schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (int64_t b = 0; b < batch; ++b) {
        for (int g = 0; g < G; ++g) {
            const size_t PN = (size_t)P * N;
            /* Sb[t]: the state token t starts from (the initial state at a start) */
            double* Sb = (double*)malloc(sizeof(double) * PN * (size_t)L);
            double* S = (double*)malloc(sizeof(double) * PN);
            double* Lam = (double*)malloc(sizeof(double) * PN);
            /* the heads of group g, in order: each adds its share of dB and dC */
            for (int h = g * hpg; h < (g + 1) * hpg; ++h) {
                int doc = 0;
                for (int64_t t = 0; t < L; ++t) {
                    int start = (t == 0);
                    if (cu && t > 0 && doc + 1 < ndocs && t == cu[doc + 1]) { ++doc; start = 1; }
                    if (start) {
                        const int st = cu ? doc : (int)b;
                        for (size_t k = 0; k < PN; ++k) S[k] = init ? init[IDX_S(st, h, 0, 0) + (int64_t)k] : 0.0;
                    }
                    memcpy(Sb + PN * (size_t)t, S, sizeof(double) * PN);
                    const double d = dt[IDX_DT(b, t, h)];
                    const double a = exp(d * A[h]);
                    for (int p = 0; p < P; ++p) {
                        const double u = d * x[IDX_X(b, t, h, p)];
                        for (int n = 0; n < N; ++n) S[p * N + n] = a * S[p * N + n] + u * B[IDX_BC(b, t, g, n)];
                    }
                }
                /* backwards in time; doc = the document of token t */
                for (int64_t t = L - 1; t >= 0; --t) {
                    while (cu && doc > 0 && t < cu[doc]) --doc;
                    const int st = cu ? doc : (int)b;
                    const int end = (t == L - 1) || (cu && doc + 1 <= ndocs && t + 1 == cu[doc + 1]);
                    if (end)   /* the final state of this sequence or document */
                        for (size_t k = 0; k < PN; ++k) Lam[k] = dfin ? dfin[IDX_S(st, h, 0, 0) + (int64_t)k] : 0.0;
                    const double d = dt[IDX_DT(b, t, h)];
                    const double a = exp(d * A[h]);
                    const double* Sprev = Sb + PN * (size_t)t;   /* S_{t-1} (or the initial state) */
                    /* Lam becomes Lam_t: add the output's use of S_t */
                    for (int p = 0; p < P; ++p)
                        for (int n = 0; n < N; ++n)
                            Lam[p * N + n] += dy[IDX_X(b, t, h, p)] * C[IDX_BC(b, t, g, n)];
                    for (int n = 0; n < N; ++n) {
                        double sc = 0.0, sb = 0.0;
                        for (int p = 0; p < P; ++p) {
                            const double scur = a * Sprev[p * N + n] + d * x[IDX_X(b, t, h, p)] * B[IDX_BC(b, t, g, n)];
                            sc += scur * dy[IDX_X(b, t, h, p)];
                            sb += Lam[p * N + n] * x[IDX_X(b, t, h, p)];
                        }
                        dC[IDX_BC(b, t, g, n)] += sc;
                        dB[IDX_BC(b, t, g, n)] += d * sb;
                    }
                    double xv = 0.0, dyx = 0.0;
                    for (int p = 0; p < P; ++p) {
                        double acc = 0.0;
                        for (int n = 0; n < N; ++n) acc += Lam[p * N + n] * B[IDX_BC(b, t, g, n)];
                        dx[IDX_X(b, t, h, p)] = d * acc + (D ? D[h] * dy[IDX_X(b, t, h, p)] : 0.0);
                        xv += x[IDX_X(b, t, h, p)] * acc;
                        dyx += dy[IDX_X(b, t, h, p)] * x[IDX_X(b, t, h, p)];
                    }
                    double ls = 0.0;
                    for (size_t k = 0; k < PN; ++k) ls += Lam[k] * Sprev[k];
                    const double dl = a * ls;
                    ddt[IDX_DT(b, t, h)] = xv + A[h] * dl;
                    dA_part[b * H + h] += d * dl;
                    dD_part[b * H + h] += dyx;
                    /* Lam becomes the adjoint of S_{t-1} (the initial state at a start) */
                    for (size_t k = 0; k < PN; ++k) Lam[k] *= a;
                    const int start = (t == 0) || (cu && t == cu[doc]);
                    if (start && dinit)
                        for (size_t k = 0; k < PN; ++k) dinit[IDX_S(st, h, 0, 0) + (int64_t)k] = Lam[k];
                }
            }
            free(Lam);
            free(S);
            free(Sb);
        }
    }
    for (int h = 0; h < H; ++h) {
        double sa = 0.0, sd = 0.0;
        for (int64_t b = 0; b < batch; ++b) {
            sa += dA_part[b * H + h];
            sd += dD_part[b * H + h];
        }
        dA[h] = sa;
        if (dD) dD[h] = sd;
    }
    free(dA_part);
    free(dD_part);
}

/* ---------------------------------------------------------------------- */
/* Quadratic (attention-like) form                                         */
/* ---------------------------------------------------------------------- */
void oracle_ssd_quadratic(int64_t batch, int64_t L, int H, int P, int N, int G,
                          const double* x, const double* dt, const double* A,
                          const double* B, const double* C, const double* D,
                          const double* init, const int32_t* cu, int ndocs,
                          double* y) {
    const int hpg = H / G;
    double* ell = (double*)malloc(sizeof(double) * (size_t)L);
    for (int64_t b = 0; b < batch; ++b) {
        for (int h = 0; h < H; ++h) {
            const int g = h / hpg;
            for (int64_t t = 0; t < L; ++t) ell[t] = dt[IDX_DT(b, t, h)] * A[h];
            for (int64_t i = 0; i < L; ++i) {
                const int di = cu ? doc_of(cu, ndocs, i) : 0;
                const int64_t dstart = cu ? cu[di] : 0;
                for (int p = 0; p < P; ++p) {
                    double acc = 0.0;
                    /* M_ij = (C_i . B_j) * L_ij * dt_j, L_ij = exp(seg(i, j)) */
                    double seg = 0.0;  /* seg(i, i) = 0, grown leftwards */
                    for (int64_t j = i; j >= dstart; --j) {
                        if (j < i) seg += ell[j + 1];
                        double cb = 0.0;
                        for (int n = 0; n < N; ++n) cb += C[IDX_BC(b, i, g, n)] * B[IDX_BC(b, j, g, n)];
                        acc += cb * exp(seg) * dt[IDX_DT(b, j, h)] * x[IDX_X(b, j, h, p)];
                    }
                    if (init) {
                        /* the initial state is h_{start-1}: decays by
                           exp(sum_{k=start..i} l_k) before C_i reads it */
                        double pre = 0.0;
                        for (int64_t k = i; k >= dstart; --k) pre += ell[k];
                        const int s = cu ? di : (int)b;
                        double cs = 0.0;
                        for (int n = 0; n < N; ++n) cs += init[IDX_S(s, h, p, n)] * C[IDX_BC(b, i, g, n)];
                        acc += exp(pre) * cs;
                    }
                    if (D) acc += D[h] * x[IDX_X(b, i, h, p)];
                    y[IDX_X(b, i, h, p)] = acc;
                }
            }
        }
    }
    free(ell);
}

/* ---------------------------------------------------------------------- */
/* Block (chunk) decomposition                                             */
/* ---------------------------------------------------------------------- */
/*
 * Tokens are cut into chunks of Q, and chunks into splits of split_len tokens
 * (split_len a multiple of Q; <= 0 or >= L: one split).  A packed document
 * boundary never needs special chunk alignment: the pieces of one chunk that
 * belong to different documents are handled as separate segments.
 *
 * Per chunk c, segment [a, e] (one document), and incoming state S0:
 *   diagonal block   y_i += sum_{j=a..i} (C_i . B_j) exp(seg(i,j)) dt_j x_j
 *   state projection y_i += exp(sum_{k=a..i} l_k) S0 C_i
 *   chunk state      S(e) = exp(sum_{k=a..e} l_k) S0
 *                           + sum_{j=a..e} exp(seg(e,j)) dt_j x_j B_j^T
 * S0 is the state carried into the chunk when the segment continues a
 * document, else the document's initial state (or zero).
 *
 * Splits: each split first runs from a zero incoming state, giving its
 * aggregate (tau_s, S_s): the state at its end and the total log-decay
 * applied to whatever entered it (-inf if a document starts inside).  The
 * incoming states are then composed left to right with
 *   (tau_1, S_1) then (tau_2, S_2)  ->  (tau_1 + tau_2, exp(tau_2) S_1 + S_2)
 * and each split is run again from its incoming state to produce y.
 */
typedef struct {
    int64_t L; int H, P, N, G, Q;
    const double *x, *dt, *A, *B, *C, *D, *init;
    const int32_t* cu; int ndocs;
} chk_ctx;

/* run tokens [t0, t1) of row b, head h from incoming state S (P x N, updated
   in place to the state at t1-1).  Writes y when y != NULL and per-document
   final states when fin != NULL.  Returns the total log-decay applied to the
   incoming state (-inf if a document starts in [t0, t1)). */
static double chk_run(const chk_ctx* c, int64_t b, int h, int64_t t0, int64_t t1, double* S,
                      int zero_start, double* y, double* fin) {
    const int64_t L = c->L; const int H = c->H, P = c->P, N = c->N, G = c->G, Q = c->Q;
    const int g = h / (H / G);
    const double *x = c->x, *dt = c->dt, *B = c->B, *C = c->C;
    double tau = 0.0;
    double* ell = (double*)malloc(sizeof(double) * Q);
    double* Snew = (double*)malloc(sizeof(double) * (size_t)P * N);
    for (int64_t c0 = t0; c0 < t1; c0 += Q) {
        const int64_t c1 = (c0 + Q < t1) ? c0 + Q : t1;
        for (int64_t t = c0; t < c1; ++t) ell[t - c0] = dt[IDX_DT(b, t, h)] * c->A[h];
        int64_t a = c0;
        while (a < c1) {
            /* segment [a, e]: up to the next document start or the chunk end */
            int64_t e = c1 - 1;
            int starts_doc = (a == 0);
            int doc = 0;
            if (c->cu) {
                doc = doc_of(c->cu, c->ndocs, a);
                starts_doc = (c->cu[doc] == a);
                if (c->cu[doc + 1] - 1 < e) e = c->cu[doc + 1] - 1;
            }
            const int sidx = c->cu ? doc : (int)b;
            if (starts_doc) {
                /* a document starts here: its initial state replaces S */
                tau = -INFINITY;
                for (int p = 0; p < P; ++p)
                    for (int n = 0; n < N; ++n)
                        S[p * N + n] = c->init ? c->init[IDX_S(sidx, h, p, n)] : 0.0;
            } else if (zero_start && a == t0) {
                /* aggregate pass: the incoming state is taken as zero */
                memset(S, 0, sizeof(double) * (size_t)P * N);
            }
            if (y) {
                for (int64_t i = a; i <= e; ++i) {
                    double pre = 0.0;  /* sum_{k=a..i} l_k */
                    for (int64_t k = i; k >= a; --k) pre += ell[k - c0];
                    for (int p = 0; p < P; ++p) {
                        double acc = 0.0, seg = 0.0;
                        for (int64_t j = i; j >= a; --j) {
                            if (j < i) seg += ell[j + 1 - c0];
                            double cb = 0.0;
                            for (int n = 0; n < N; ++n) cb += C[IDX_BC(b, i, g, n)] * B[IDX_BC(b, j, g, n)];
                            acc += cb * exp(seg) * dt[IDX_DT(b, j, h)] * x[IDX_X(b, j, h, p)];
                        }
                        double cs = 0.0;
                        for (int n = 0; n < N; ++n) cs += S[p * N + n] * C[IDX_BC(b, i, g, n)];
                        acc += exp(pre) * cs;
                        if (c->D) acc += c->D[h] * x[IDX_X(b, i, h, p)];
                        y[IDX_X(b, i, h, p)] = acc;
                    }
                }
            }
            /* chunk (segment) state at e */
            double tot = 0.0;
            for (int64_t k = e; k >= a; --k) tot += ell[k - c0];
            for (int p = 0; p < P; ++p)
                for (int n = 0; n < N; ++n) Snew[p * N + n] = exp(tot) * S[p * N + n];
            double suf = 0.0;  /* seg(e, j) = sum_{k=j+1..e} l_k */
            for (int64_t j = e; j >= a; --j) {
                if (j < e) suf += ell[j + 1 - c0];
                const double w = exp(suf) * dt[IDX_DT(b, j, h)];
                for (int p = 0; p < P; ++p) {
                    const double u = w * x[IDX_X(b, j, h, p)];
                    for (int n = 0; n < N; ++n) Snew[p * N + n] += u * B[IDX_BC(b, j, g, n)];
                }
            }
            memcpy(S, Snew, sizeof(double) * (size_t)P * N);
            tau += tot;
            const int doc_end = (e == L - 1) || (c->cu && e + 1 == c->cu[doc + 1]);
            if (fin && doc_end)
                for (int p = 0; p < P; ++p)
                    for (int n = 0; n < N; ++n) fin[IDX_S(sidx, h, p, n)] = S[p * N + n];
            a = e + 1;
        }
    }
    free(ell);
    free(Snew);
    return tau;
}

void oracle_ssd_chunked(int64_t batch, int64_t L, int H, int P, int N, int G,
                        const double* x, const double* dt, const double* A,
                        const double* B, const double* C, const double* D,
                        const double* init, const int32_t* cu, int ndocs,
                        int Q, int64_t split_len, double* y, double* final_states) {
    chk_ctx c = {L, H, P, N, G, Q, x, dt, A, B, C, D, init, cu, ndocs};
    if (split_len <= 0 || split_len > L) split_len = L;
    const int64_t nsplit = (L + split_len - 1) / split_len;
    const size_t PN = (size_t)P * N;
    double* agg = (double*)malloc(sizeof(double) * PN * nsplit);
    double* tau = (double*)malloc(sizeof(double) * nsplit);
    double* Sin = (double*)malloc(sizeof(double) * PN);
    for (int64_t b = 0; b < batch; ++b) {
        for (int h = 0; h < H; ++h) {
            /* pass 1: split aggregates from a zero incoming state */
            for (int64_t s = 0; s < nsplit; ++s) {
                const int64_t t0 = s * split_len, t1 = (t0 + split_len < L) ? t0 + split_len : L;
                tau[s] = chk_run(&c, b, h, t0, t1, agg + s * PN, 1, NULL, NULL);
            }
            /* pass 2: compose incoming states, then run each split for y */
            memset(Sin, 0, sizeof(double) * PN);
            for (int64_t s = 0; s < nsplit; ++s) {
                const int64_t t0 = s * split_len, t1 = (t0 + split_len < L) ? t0 + split_len : L;
                double* St = (double*)malloc(sizeof(double) * PN);
                memcpy(St, Sin, sizeof(double) * PN);
                chk_run(&c, b, h, t0, t1, St, 0, y, final_states);
                free(St);
                const double e = exp(tau[s]);
                for (size_t k = 0; k < PN; ++k) Sin[k] = e * Sin[k] + agg[s * PN + k];
            }
        }
    }
    free(agg); free(tau); free(Sin);
}

/* ---------------------------------------------------------------------- */
/* Segsum                                                                  */
/* ---------------------------------------------------------------------- */
/* ell: nrows x len (fp64).  seg: nrows x len x len; seg[i][j] for j <= i is
   sum_{k=j+1..i} ell_k accumulated from the diagonal leftwards; -inf above. */
void oracle_segsum(const double* ell, int64_t nrows, int len, double* seg) {
    for (int64_t r = 0; r < nrows; ++r) {
        const double* l = ell + r * len;
        double* o = seg + r * (int64_t)len * len;
        for (int i = 0; i < len; ++i) {
            double acc = 0.0;
            for (int j = i; j >= 0; --j) {
                if (j < i) acc += l[j + 1];
                o[(int64_t)i * len + j] = acc;
            }
            for (int j = i + 1; j < len; ++j) o[(int64_t)i * len + j] = -INFINITY;
        }
    }
}

/* fp32 diff segsum comparator: Kogge-Stone inclusive cumsum, then
   cum_i - cum_j below the diagonal, -inf above. */
void oracle_diff_segsum_f32(const float* ell, int64_t nrows, int len, float* seg) {
    float* cum = (float*)malloc(sizeof(float) * len);
    float* nxt = (float*)malloc(sizeof(float) * len);
    for (int64_t r = 0; r < nrows; ++r) {
        for (int i = 0; i < len; ++i) cum[i] = ell[r * len + i];
        for (int d = 1; d < len; d <<= 1) {
            for (int i = 0; i < len; ++i) nxt[i] = (i >= d) ? cum[i] + cum[i - d] : cum[i];
            memcpy(cum, nxt, sizeof(float) * len);
        }
        float* o = seg + r * (int64_t)len * len;
        for (int i = 0; i < len; ++i)
            for (int j = 0; j < len; ++j)
                o[(int64_t)i * len + j] = (j <= i) ? cum[i] - cum[j] : -INFINITY;
    }
    free(cum); free(nxt);
}
