/*
 * CPU oracle for the Mamba-2 selective-state recurrence.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  Only the tests, the smoke
 * check and the benchmark's CPU-baseline leg may load this code.  It shares
 * no code, header, table or helper with the CUDA library.
 *
 * Plain, slow, obviously correct: scalar loops in fp64 (compiled without
 * FMA contraction or fast-math), one function per form of the computation.
 * Independent (request, head) pairs are spread over threads with OpenMP;
 * that changes no arithmetic, since each pair's loop is sequential.
 *
 * The recurrence (Mamba-2 selective state space, as used by all three
 * pages: Mamba Streaming State That Survives
 * Chunking / Separate Mamba-2 algebra from kernel behavior; Why Speculative
 * Decoding Slows Hybrid Mamba Models / The Fix):
 *
 *   dA_t      = exp(dt_t * A_h)
 *   h_t[p,n]  = dA_t * h_{t-1}[p,n] + dt_t * x_t[p] * B_t[g(h),n]
 *   y_t[p]    = sum_n C_t[g(h),n] * h_t[p,n] + D_h * x_t[p]
 *
 * Each token decays the previous state and then adds its own contribution
 * (The Fix); the output reads the state after the token is applied.  Heads map to
 * groups in contiguous blocks, g(h) = h / (H / G).
 *
 * The same source builds two libraries: the parity oracle in fp64 (the
 * default) and, with -DORACLE_F32, an instantiation whose every value and
 * accumulator is fp32 -- the same loops in the same order, used only as the
 * CPU speed baseline (a fast CPU code would hold fp32, as the GPU does).
 *
 * Every function that produces outputs y can also produce ycond (pass NULL
 * to skip it): for each output element, sum_n |C[n] h[p,n]| + |D x[p]| with
 * h the state after that token -- the size of the terms whose sum is y.
 * A result computed in fp32 can be expected to carry an error relative to
 * this scale, not to |y|, which cancellation in the sum over n can make
 * arbitrarily small; the parity tests take their relative tolerance
 * against it.
 *
 * Functions:
 *   oracle_scan_head      sequential recurrence of one (sequence, head)
 *   oracle_decode_step    one token for a batch of requests
 *   oracle_verify_copy    T+1 tokens, a full state copy after each
 *   oracle_replay_head    outputs from checkpoint + input log (closed form)
 *   oracle_verify_replay  the same over a batch
 *   oracle_fold           apply log entries then accepted tokens to the checkpoint
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_ABI_VERSION 2

#ifdef ORACLE_F32
typedef float real;
#define EXP expf
#define ABS fabsf
#else
typedef double real;
#define EXP exp
#define ABS fabs
#endif

int oracle_abi_version(void) { return ORACLE_ABI_VERSION; }
int oracle_real_bytes(void) { return (int)sizeof(real); }

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads of the parallel loops that follow (timing only; no effect on results). */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/*
 * Sequential recurrence for one (sequence, head) over L tokens.
 *   state [P][N]     in: state before the first token, out: after the last
 *   x     token t at x  + t*xs,  P values
 *   dt    token t at dt + t*dts
 *   B, C  token t at B  + t*bcs, N values (this head's group)
 *   y     token t at y  + t*ys,  P values; may be NULL (state only)
 *   ycond as y: the condition scale of each output; may be NULL
 */
void oracle_scan_head(int P, int N, long L, real A, real D,
                      const real *x, long xs, const real *dt, long dts,
                      const real *B, const real *C, long bcs,
                      real *state, real *y, long ys, real *ycond)
{
    for (long t = 0; t < L; t++) {
        const real *xt = x + t * xs;
        const real *Bt = B + t * bcs;
        const real *Ct = C + t * bcs;
        const real dtt = dt[t * dts];
        const real dA = EXP(dtt * A);
        for (int p = 0; p < P; p++)
            for (int n = 0; n < N; n++)
                state[p * N + n] = dA * state[p * N + n] + dtt * xt[p] * Bt[n];
        if (y) {
            for (int p = 0; p < P; p++) {
                real acc = 0;
                for (int n = 0; n < N; n++)
                    acc += Ct[n] * state[p * N + n];
                y[t * ys + p] = acc + D * xt[p];
            }
        }
        if (ycond) {
            for (int p = 0; p < P; p++) {
                real acc = 0;
                for (int n = 0; n < N; n++)
                    acc += ABS(Ct[n] * state[p * N + n]);
                ycond[t * ys + p] = acc + ABS(D * xt[p]);
            }
        }
    }
}

/*
 * One decode token for R requests (batched single-token update).
 *   state [R][H][P][N] in/out
 *   x [R][H][P], dt [R][H], B, C [R][G][N], A, D [H], y [R][H][P]
 *   ycond [R][H][P] or NULL
 */
void oracle_decode_step(int R, int H, int P, int N, int G, real *state,
                        const real *x, const real *dt, const real *B, const real *C,
                        const real *A, const real *D, real *y, real *ycond)
{
    const int hpg = H / G;
#pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < R; r++)
        for (int h = 0; h < H; h++) {
            const int g = h / hpg;
            oracle_scan_head(P, N, 1, A[h], D[h],
                             x + ((long)r * H + h) * P, 0,
                             dt + (long)r * H + h, 0,
                             B + ((long)r * G + g) * N, C + ((long)r * G + g) * N, 0,
                             state + ((long)r * H + h) * P * N,
                             y + ((long)r * H + h) * P, 0,
                             ycond ? ycond + ((long)r * H + h) * P : NULL);
        }
}

/*
 * Speculative verify with per-draft state copies (Why Speculative Decoding
 * Slows Hybrid Mamba Models / The Problem: one full state copy is kept per
 * draft so that a rejected draft can be undone).  Request r walks its T1 = T+1 tokens from its
 * current state; after token j the full state is saved as snapshot j.
 *   state [R][H][P][N]         read only
 *   x [R][T1][H][P], dt [R][T1][H], B, C [R][T1][G][N]
 *   snap [T1][R][H][P][N]      out
 *   y [R][T1][H][P]            out
 *   ycond [R][T1][H][P]        out, or NULL
 */
void oracle_verify_copy(int R, int T1, int H, int P, int N, int G,
                        const real *state, const real *x, const real *dt,
                        const real *B, const real *C, const real *A, const real *D,
                        real *snap, real *y, real *ycond)
{
    const int hpg = H / G;
    const long S = (long)P * N;
#pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < R; r++)
        for (int h = 0; h < H; h++) {
            const int g = h / hpg;
            real *cur = (real *)malloc(sizeof(real) * S);
            memcpy(cur, state + ((long)r * H + h) * S, sizeof(real) * S);
            for (int j = 0; j < T1; j++) {
                const long tok = (long)r * T1 + j;
                oracle_scan_head(P, N, 1, A[h], D[h],
                                 x + (tok * H + h) * P, 0, dt + tok * H + h, 0,
                                 B + (tok * G + g) * N, C + (tok * G + g) * N, 0,
                                 cur, y + (tok * H + h) * P, 0,
                                 ycond ? ycond + (tok * H + h) * P : NULL);
                memcpy(snap + (((long)j * R + r) * H + h) * S, cur, sizeof(real) * S);
            }
            free(cur);
        }
}

/*
 * ReplaySSM output for one (request, head), closed form (Why Speculative
 * Decoding Slows Hybrid Mamba Models / The Fix: the unrolled update is the
 * decayed checkpoint plus every logged token's term, each decayed by the
 * time elapsed since that token).
 *
 * u_0 .. u_{k+n_tok-1} are the k logged tokens followed by the n_tok step
 * tokens.  For step token j, the tokens applied so far are u_0 .. u_{m-1}
 * with m = k + j + 1, and
 *
 *   y_j[p] = exp(A * sum_{r<m} dt_r) * (C_j . hc[p,:])
 *          + sum_{s<m} exp(A * sum_{s<r<m} dt_r) * dt_s * (C_j . B_s) * x_s[p]
 *          + D * x_j[p]
 *
 *   hc  [P][N]                  checkpoint (read only)
 *   ux  [k+n_tok][P], udt [k+n_tok], uB [k+n_tok][N]   the token sequence u
 *   Cq  [n_tok][N]              C of the step tokens
 *   y   [n_tok][P]              out
 *   ycond [n_tok][P]            out, or NULL: the condition scale of y_j,
 *                               which needs the state after each token, so
 *                               it walks the tokens sequentially from hc (for
 *                               the scale only; y above is the closed form)
 */
void oracle_replay_head(int P, int N, int k, int n_tok, real A, real D,
                        const real *hc, const real *ux, const real *udt,
                        const real *uB, const real *Cq, real *y, real *ycond)
{
    real *cb = (real *)malloc(sizeof(real) * (k + n_tok));
    real *w = (real *)malloc(sizeof(real) * (k + n_tok));
    for (int j = 0; j < n_tok; j++) {
        const int m = k + j + 1;
        const real *Cj = Cq + (long)j * N;
        const real *xj = ux + (long)(k + j) * P;
        /* decay weight of each applied token: time elapsed after it */
        real after = 0;
        for (int s = m - 1; s >= 0; s--) {
            real dot = 0;
            for (int n = 0; n < N; n++)
                dot += Cj[n] * uB[(long)s * N + n];
            cb[s] = dot;
            w[s] = EXP(A * after) * udt[s];
            after += udt[s];
        }
        const real decay_all = EXP(A * after);   /* after == sum of all m dt */
        for (int p = 0; p < P; p++) {
            real ch = 0;
            for (int n = 0; n < N; n++)
                ch += Cj[n] * hc[(long)p * N + n];
            real acc = decay_all * ch;
            for (int s = 0; s < m; s++)
                acc += w[s] * cb[s] * ux[(long)s * P + p];
            y[(long)j * P + p] = acc + D * xj[p];
        }
    }
    free(cb);
    free(w);
    if (ycond) {
        real *h = (real *)malloc(sizeof(real) * (long)P * N);
        memcpy(h, hc, sizeof(real) * (long)P * N);
        for (int s = 0; s < k + n_tok; s++) {
            const int j = s - k;   /* a step token from s = k on */
            oracle_scan_head(P, N, 1, A, D, ux + (long)s * P, 0, udt + s, 0, uB + (long)s * N,
                             j >= 0 ? Cq + (long)j * N : uB + (long)s * N, 0, h, NULL, 0,
                             j >= 0 ? ycond + (long)j * P : NULL);
        }
        free(h);
    }
}

/*
 * ReplaySSM verify for R requests.
 *   ckpt [R][H][P][N]                         checkpoints (read only)
 *   log_len [R]                               logged tokens per request
 *   lx [R][Wc][H][P], ldt [R][Wc][H], lB [R][Wc][G][N]   logs (capacity Wc)
 *   x [R][T1][H][P], dt [R][T1][H], B, C [R][T1][G][N]   step tokens
 *   y [R][T1][H][P]                           out
 */
void oracle_verify_replay(int R, int T1, int H, int P, int N, int G, int Wc,
                          const real *ckpt, const int *log_len,
                          const real *lx, const real *ldt, const real *lB,
                          const real *x, const real *dt, const real *B, const real *C,
                          const real *A, const real *D, real *y, real *ycond)
{
    const int hpg = H / G;
    const long S = (long)P * N;
#pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < R; r++)
        for (int h = 0; h < H; h++) {
            const int g = h / hpg;
            const int k = log_len[r];
            const int m = k + T1;
            real *ux = (real *)malloc(sizeof(real) * (long)m * P);
            real *udt = (real *)malloc(sizeof(real) * m);
            real *uB = (real *)malloc(sizeof(real) * (long)m * N);
            real *Cq = (real *)malloc(sizeof(real) * (long)T1 * N);
            real *yh = (real *)malloc(sizeof(real) * (long)T1 * P);
            real *ch = ycond ? (real *)malloc(sizeof(real) * (long)T1 * P) : NULL;
            for (int s = 0; s < k; s++) {
                const long e = (long)r * Wc + s;
                memcpy(ux + (long)s * P, lx + (e * H + h) * P, sizeof(real) * P);
                udt[s] = ldt[e * H + h];
                memcpy(uB + (long)s * N, lB + (e * G + g) * N, sizeof(real) * N);
            }
            for (int j = 0; j < T1; j++) {
                const long tok = (long)r * T1 + j;
                memcpy(ux + (long)(k + j) * P, x + (tok * H + h) * P, sizeof(real) * P);
                udt[k + j] = dt[tok * H + h];
                memcpy(uB + (long)(k + j) * N, B + (tok * G + g) * N, sizeof(real) * N);
                memcpy(Cq + (long)j * N, C + (tok * G + g) * N, sizeof(real) * N);
            }
            oracle_replay_head(P, N, k, T1, A[h], D[h], ckpt + ((long)r * H + h) * S,
                               ux, udt, uB, Cq, yh, ch);
            for (int j = 0; j < T1; j++) {
                memcpy(y + (((long)r * T1 + j) * H + h) * P, yh + (long)j * P, sizeof(real) * P);
                if (ch)
                    memcpy(ycond + (((long)r * T1 + j) * H + h) * P, ch + (long)j * P, sizeof(real) * P);
            }
            free(ux); free(udt); free(uB); free(Cq); free(yh); free(ch);
        }
}

/*
 * Fold: write the checkpoint forward through the logged tokens and then the
 * first c[r] step tokens, sequentially (The Fix: the full state is written
 * only when the log window is full).  Requests with fold[r] == 0 are untouched.
 *   ckpt [R][H][P][N] in/out; log arrays as in oracle_verify_replay;
 *   step tokens x [R][T1][H][P], dt [R][T1][H], B [R][T1][G][N]
 *   (C is not needed: no output is produced).
 */
void oracle_fold(int R, int T1, int H, int P, int N, int G, int Wc,
                 real *ckpt, const int *log_len, const int *c, const int *fold,
                 const real *lx, const real *ldt, const real *lB,
                 const real *x, const real *dt, const real *B, const real *A)
{
    const int hpg = H / G;
    const long S = (long)P * N;
#pragma omp parallel for collapse(2) schedule(static)
    for (int r = 0; r < R; r++)
        for (int h = 0; h < H; h++) {
            if (!fold[r])
                continue;
            const int g = h / hpg;
            real *st = ckpt + ((long)r * H + h) * S;
            const long e0 = (long)r * Wc;
            oracle_scan_head(P, N, log_len[r], A[h], 0,
                             lx + (e0 * H + h) * P, (long)H * P, ldt + e0 * H + h, H,
                             lB + (e0 * G + g) * N, lB + (e0 * G + g) * N, (long)G * N,
                             st, NULL, 0, NULL);
            const long t0 = (long)r * T1;
            oracle_scan_head(P, N, c[r], A[h], 0,
                             x + (t0 * H + h) * P, (long)H * P, dt + t0 * H + h, H,
                             B + (t0 * G + g) * N, B + (t0 * G + g) * N, (long)G * N,
                             st, NULL, 0, NULL);
        }
}
