/*
 * moments_oracle.c -- fp64 CPU oracle for the physical-frame state-moments operator.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and bench.py's
 * cpu_baseline / reference leg may load or run this file.  It shares no code,
 * header, table or helper with the CUDA path in state_space_model_chunk_gb300/.
 *
 * What it computes (burn-mamba, "mamba3/moments/backward.rs", module header
 * "Gradient math"; "mamba3/moments/recalculated.rs", moments_phys_fwd,
 * chunk_decay, chunk_states, rotate_chunk, chunk_mask, quat_mul_prim):
 *
 *   h_{-1} = initial[b,h]                                   (p x r)
 *   h_t    = exp(da[b,t,h]) * h_{t-1} + W_t,  W_t = sum_c xhat[b,t,c,h,:] (x) bhat[b,t,c,h,:]
 *   c_t    = derot_t(h_t)         rotation acts on the r axis of every row p
 *   m2    += sum_p c_t[p,:]^T c_t[p,:]      m1 += sum_p c_t[p,:]       for t < valid_len[b]
 *
 * This is the plain definition the chunked form reaches exactly: inside a chunk
 * the inclusive cumsum a_t of da gives d_t = exp(a_t) and L[t,j] = exp(a_t - a_j)
 * with L[t,t] = 1, so h~[t] = d_t h_- + sum_{j<=t} L[t,j] W_j is the same
 * recurrence unrolled, and chunk_len does not change the result.
 *
 * Backward: plain reverse-mode differentiation of the recurrence above, token by
 * token, with the moments VJP d_c = c (D + D^T) + 1_p (x) d_m1 ("backward.rs"
 * header, first bullet), the rotation VJPs of the header's second bullet, and the
 * write VJPs d_xhat = g . bhat, d_bhat = g^T . xhat (header, fourth bullet).
 * d_da is the direct derivative of h_t = e^{da_t} h_{t-1} + W_t, which the
 * header's reverse-cumsum identity rewrites chunkwise.
 *
 * All arithmetic is fp64.  The (b,h) pairs are independent and run under OpenMP.
 * Readings of points the pages leave open (one valid_len per batch row; m1 of
 * shape [b,h,r]; angles width rope_dim/2; half-split pairs (i, i + r/2)) are the
 * ones the rest of the pages support and are listed in the design notes.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_ROT_NONE = 0, OR_ROT_PAIRWISE = 1, OR_ROT_HALF = 2, OR_ROT_QUAT = 3 };

typedef struct {
    int64_t b, s, C, h, p, r;
    int rot;          /* OR_ROT_* */
    int64_t rope_dim; /* complex kinds: rotated width (even); angles per token = rope_dim/2 */
    int64_t J;        /* quaternion blocks (4J <= r) */
} or_dims;

/* ---- Hamilton product on (w,x,y,z) ("recalculated.rs", quat_mul_prim) ---- */
static void qmul(const double a[4], const double b[4], double out[4]) {
    out[0] = a[0] * b[0] - a[1] * b[1] - a[2] * b[2] - a[3] * b[3];
    out[1] = a[0] * b[1] + a[1] * b[0] + a[2] * b[3] - a[3] * b[2];
    out[2] = a[0] * b[2] - a[1] * b[3] + a[2] * b[0] + a[3] * b[1];
    out[3] = a[0] * b[3] + a[1] * b[2] - a[2] * b[1] + a[3] * b[0];
}

/* ---- rotation of one state row ("recalculated.rs", rotate_chunk, chunk_cos_sin) ----
 * transpose = 0: de-rotation to the physical frame, R(-theta) per complex pair,
 *                left multiplication by Q per quaternion block.
 * transpose = 1: its transpose, R(+theta) / left multiplication by conj(Q).
 * ang: the token's rope_dim/2 cumulative angles; q: its J cumulative quaternions.
 * Dimensions outside the rotated set pass through unchanged. */
static void pair_index(const or_dims* d, int64_t i, int64_t* ix, int64_t* iy) {
    if (d->rot == OR_ROT_PAIRWISE) { *ix = 2 * i; *iy = 2 * i + 1; }
    else { *ix = i; *iy = i + d->r / 2; }                 /* half-split: distance r/2 */
}

static void rotate_row(const or_dims* d, const double* v, double* out,
                       const double* ang, const double* q, int transpose) {
    memcpy(out, v, sizeof(double) * (size_t)d->r);
    if (d->rot == OR_ROT_PAIRWISE || d->rot == OR_ROT_HALF) {
        for (int64_t i = 0; i < d->rope_dim / 2; ++i) {
            int64_t ix, iy;
            pair_index(d, i, &ix, &iy);
            double phi = transpose ? ang[i] : -ang[i];
            double cs = cos(phi), sn = sin(phi);
            out[ix] = cs * v[ix] - sn * v[iy];
            out[iy] = sn * v[ix] + cs * v[iy];
        }
    } else if (d->rot == OR_ROT_QUAT) {
        for (int64_t k = 0; k < d->J; ++k) {
            double Q[4] = {q[4 * k], q[4 * k + 1], q[4 * k + 2], q[4 * k + 3]};
            if (transpose) { Q[1] = -Q[1]; Q[2] = -Q[2]; Q[3] = -Q[3]; }
            qmul(Q, v + 4 * k, out + 4 * k);
        }
    }
}

/* index helpers, all tensors row-major */
#define IX_X(d, bb, t, c, hh, pp) (((((bb) * (d)->s + (t)) * (d)->C + (c)) * (d)->h + (hh)) * (d)->p + (pp))
#define IX_B(d, bb, t, c, hh, rr) (((((bb) * (d)->s + (t)) * (d)->C + (c)) * (d)->h + (hh)) * (d)->r + (rr))
#define IX_DA(d, bb, t, hh) ((((bb) * (d)->s + (t)) * (d)->h) + (hh))

static int64_t rot_width(const or_dims* d) {
    if (d->rot == OR_ROT_PAIRWISE || d->rot == OR_ROT_HALF) return d->rope_dim / 2;
    if (d->rot == OR_ROT_QUAT) return 4 * d->J;
    return 0;
}
static const double* rot_at(const or_dims* d, const double* rot, int64_t bb, int64_t t, int64_t hh) {
    int64_t w = rot_width(d);
    if (w == 0 || rot == NULL) return NULL;
    return rot + (((bb * d->s + t) * d->h) + hh) * w;
}

static int check_dims(const or_dims* d) {
    if (d->b < 0 || d->s < 0 || d->C < 1 || d->h < 1 || d->p < 1 || d->r < 1) return 1;
    if (d->rot == OR_ROT_PAIRWISE && (d->rope_dim % 2 || d->rope_dim > d->r || d->rope_dim < 0)) return 1;
    if (d->rot == OR_ROT_HALF && (d->rope_dim % 2 || d->r % 2 || d->rope_dim / 2 > d->r / 2 || d->rope_dim < 0)) return 1;
    if (d->rot == OR_ROT_QUAT && (d->J < 0 || 4 * d->J > d->r)) return 1;
    if (d->rot < 0 || d->rot > 3) return 1;
    return 0;
}

/* Advance one token: h <- exp(da) h + sum_c xhat (x) bhat  (the recurrence above). */
static void step_state(const or_dims* d, const double* xhat, const double* bhat, const double* da,
                       int64_t bb, int64_t t, int64_t hh, const double* hprev, double* hout) {
    const int64_t p = d->p, r = d->r;
    double e = exp(da[IX_DA(d, bb, t, hh)]);
    for (int64_t i = 0; i < p; ++i)
        for (int64_t j = 0; j < r; ++j) hout[i * r + j] = e * hprev[i * r + j];
    for (int64_t c = 0; c < d->C; ++c)
        for (int64_t i = 0; i < p; ++i) {
            double xv = xhat[IX_X(d, bb, t, c, hh, i)];
            for (int64_t j = 0; j < r; ++j) hout[i * r + j] += xv * bhat[IX_B(d, bb, t, c, hh, j)];
        }
}

/* ------------------------------------------------------------------ forward */
int moments_oracle_fwd(const double* xhat, const double* bhat, const double* da, const double* rot,
                       const double* initial, const int64_t* valid_len,
                       int64_t b, int64_t s, int64_t C, int64_t h, int64_t p, int64_t r,
                       int rot_kind, int64_t rope_dim, int64_t J, int64_t bh_begin, int64_t bh_end,
                       double* m2, double* m1) {
    or_dims d = {b, s, C, h, p, r, rot_kind, rope_dim, J};
    if (check_dims(&d)) return 1;
    if (bh_end < 0 || bh_end > b * h) bh_end = b * h;
    int64_t fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : fail)
    for (int64_t bh = bh_begin; bh < bh_end; ++bh) {
        int64_t bb = bh / h, hh = bh % h;
        double* hs = (double*)malloc(sizeof(double) * (size_t)(2 * p * r + 2 * r));
        if (!hs) { fail += 1; continue; }
        double* cur = hs;            /* h_t */
        double* nxt = hs + p * r;    /* h_{t+1} scratch */
        double* crow = hs + 2 * p * r;
        double* tmp = crow + r;
        (void)tmp;
        double* M2 = m2 + bh * r * r;
        double* M1 = m1 + bh * r;
        memset(M2, 0, sizeof(double) * (size_t)(r * r));
        memset(M1, 0, sizeof(double) * (size_t)r);
        memcpy(cur, initial + bh * p * r, sizeof(double) * (size_t)(p * r));
        int64_t T = valid_len[bb] < s ? valid_len[bb] : s;
        if (T < 0) T = 0;
        for (int64_t t = 0; t < T; ++t) {
            step_state(&d, xhat, bhat, da, bb, t, hh, cur, nxt);
            double* sw = cur; cur = nxt; nxt = sw;
            const double* rt = rot_at(&d, rot, bb, t, hh);
            for (int64_t i = 0; i < p; ++i) {
                rotate_row(&d, cur + i * r, crow, rt, rt, 0);
                for (int64_t a = 0; a < r; ++a) {
                    M1[a] += crow[a];
                    for (int64_t c2 = 0; c2 < r; ++c2) M2[a * r + c2] += crow[a] * crow[c2];
                }
            }
        }
        free(hs);
    }
    return fail ? 2 : 0;
}

/* ----------------------------------------------------------------- backward */
int moments_oracle_bwd(const double* xhat, const double* bhat, const double* da, const double* rot,
                       const double* initial, const int64_t* valid_len,
                       int64_t b, int64_t s, int64_t C, int64_t h, int64_t p, int64_t r,
                       int rot_kind, int64_t rope_dim, int64_t J, int64_t bh_begin, int64_t bh_end,
                       const double* d_m2, const double* d_m1,
                       double* d_xhat, double* d_bhat, double* d_da, double* d_rot, double* d_initial) {
    or_dims d = {b, s, C, h, p, r, rot_kind, rope_dim, J};
    if (check_dims(&d)) return 1;
    if (bh_end < 0 || bh_end > b * h) bh_end = b * h;
    const int64_t rw = rot_width(&d);
    int64_t fail = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(+ : fail)
    for (int64_t bh = bh_begin; bh < bh_end; ++bh) {
        int64_t bb = bh / h, hh = bh % h;
        int64_t T = valid_len[bb] < s ? valid_len[bb] : s;
        if (T < 0) T = 0;
        /* zero this (b,h)'s slice of every gradient; positions t >= T stay zero
         * ("backward.rs" header: chunks past valid_len get zero gradients) */
        for (int64_t t = 0; t < s; ++t) {
            for (int64_t c = 0; c < C; ++c) {
                for (int64_t i = 0; i < p; ++i) d_xhat[IX_X(&d, bb, t, c, hh, i)] = 0.0;
                for (int64_t j = 0; j < r; ++j) d_bhat[IX_B(&d, bb, t, c, hh, j)] = 0.0;
            }
            d_da[IX_DA(&d, bb, t, hh)] = 0.0;
            if (rw) for (int64_t k = 0; k < rw; ++k) d_rot[(((bb * s + t) * h) + hh) * rw + k] = 0.0;
        }
        /* trajectory h_0 .. h_{T-1} for this (b,h) only */
        double* traj = (double*)malloc(sizeof(double) * (size_t)((T + 1) * p * r));
        double* work = (double*)malloc(sizeof(double) * (size_t)(2 * p * r + 6 * r + r * r));
        if (!traj || !work) { free(traj); free(work); fail += 1; continue; }
        double* H0 = traj;                       /* h_{-1} = initial */
        memcpy(H0, initial + bh * p * r, sizeof(double) * (size_t)(p * r));
        for (int64_t t = 0; t < T; ++t)
            step_state(&d, xhat, bhat, da, bb, t, hh, traj + t * p * r, traj + (t + 1) * p * r);
        double* g = work;                         /* running cotangent of h_t */
        double* gtmp = work + p * r;
        double* crow = gtmp + p * r;
        double* dc = crow + r;
        double* back = dc + r;
        double* Dsym = back + r + 3 * r;
        for (int64_t a = 0; a < r; ++a)
            for (int64_t c2 = 0; c2 < r; ++c2)
                Dsym[a * r + c2] = d_m2[bh * r * r + a * r + c2] + d_m2[bh * r * r + c2 * r + a];
        memset(g, 0, sizeof(double) * (size_t)(p * r));
        for (int64_t t = T - 1; t >= 0; --t) {
            const double* ht = traj + (t + 1) * p * r;     /* h_t */
            const double* hp = traj + t * p * r;           /* h_{t-1} */
            const double* rt = rot_at(&d, rot, bb, t, hh);
            double* drt = rw ? d_rot + (((bb * s + t) * h) + hh) * rw : NULL;
            for (int64_t i = 0; i < p; ++i) {
                /* moments VJP on row i */
                rotate_row(&d, ht + i * r, crow, rt, rt, 0);
                for (int64_t c2 = 0; c2 < r; ++c2) {
                    double acc = d_m1[bh * r + c2];
                    for (int64_t a = 0; a < r; ++a) acc += crow[a] * Dsym[a * r + c2];
                    dc[c2] = acc;
                }
                /* rotation parameter VJP */
                if (d.rot == OR_ROT_PAIRWISE || d.rot == OR_ROT_HALF) {
                    for (int64_t k = 0; k < rope_dim / 2; ++k) {
                        int64_t ix, iy;
                        pair_index(&d, k, &ix, &iy);
                        drt[k] += dc[ix] * crow[iy] - dc[iy] * crow[ix];
                    }
                } else if (d.rot == OR_ROT_QUAT) {
                    for (int64_t k = 0; k < J; ++k) {
                        const double* hb = ht + i * r + 4 * k;
                        double hc[4] = {hb[0], -hb[1], -hb[2], -hb[3]};
                        double prod[4];
                        qmul(dc + 4 * k, hc, prod);
                        for (int q = 0; q < 4; ++q) drt[4 * k + q] += prod[q];
                    }
                }
                /* cotangent back to the cache frame, accumulated into g */
                rotate_row(&d, dc, back, rt, rt, 1);
                for (int64_t a = 0; a < r; ++a) g[i * r + a] += back[a];
            }
            /* g is now the full cotangent of h_t */
            for (int64_t c = 0; c < C; ++c) {
                for (int64_t i = 0; i < p; ++i) {
                    double acc = 0.0;
                    for (int64_t a = 0; a < r; ++a) acc += g[i * r + a] * bhat[IX_B(&d, bb, t, c, hh, a)];
                    d_xhat[IX_X(&d, bb, t, c, hh, i)] = acc;
                }
                for (int64_t a = 0; a < r; ++a) {
                    double acc = 0.0;
                    for (int64_t i = 0; i < p; ++i) acc += g[i * r + a] * xhat[IX_X(&d, bb, t, c, hh, i)];
                    d_bhat[IX_B(&d, bb, t, c, hh, a)] = acc;
                }
            }
            double e = exp(da[IX_DA(&d, bb, t, hh)]);
            double dot = 0.0;
            for (int64_t k = 0; k < p * r; ++k) dot += g[k] * hp[k];
            d_da[IX_DA(&d, bb, t, hh)] = e * dot;
            for (int64_t k = 0; k < p * r; ++k) g[k] *= e;
        }
        memcpy(d_initial + bh * p * r, g, sizeof(double) * (size_t)(p * r));
        free(traj);
        free(work);
    }
    return fail ? 2 : 0;
}

int moments_oracle_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
