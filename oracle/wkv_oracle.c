/*
 * wkv_oracle.c -- plain, slow, float64 CPU reference of the WKV operator.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library
 * and its Python binding) may call, link or load this file.  It is used by
 * the tests, by __graft_entry__.smoke() and by bench.py's CPU baseline leg.
 * It shares no code, header, table or helper with the CUDA sources.
 *
 * What it computes (sources, by page title and section):
 *
 *  - "RWKV解读：在Transformer的时代的新RNN" (segmentfault), section
 *    "3、RWKV的网络架构", equation (8): the time-mixing "attention" wkv.  The
 *    page says the absolute-position bias of AFT is replaced by a relative
 *    one driven by a single trained vector w, the current position gets its
 *    own parameter u, and that eq. (8) can be written recursively.
 *  - "RWKV についての調査記録" (qiita), section "wkvとは": wkv is a weighted
 *    average of v with weights from k; the current v receives a bonus u;
 *    past v are decayed more the further back they are, through one
 *    channel-wise decay vector w; all channels are computed independently.
 *  - Same page, section "Trainingについて": all parameters get gradients
 *    from the loss, so w, u, k and v all need gradients.
 *  - "RWKV解读" section "3、RWKV的网络架构", equations (7) and (9): the
 *    token shift (input is a weighted sum of the current and the previous
 *    token) and the sigmoid(r) gate on the time-mixing output.
 *  - "介绍RWKV – 具有Transformer优势的RNN" (xiaozhuai), section
 *    "RWKV作为RNN和transformer的结合体", and qiita "RWKVとは？": in
 *    inference the layer takes a token and a state and returns an output
 *    and a new state (the decode step).
 *
 * The pages lost the bodies of every equation, so the exact form used here
 * is the standard RWKV-4 definition, which matches every property the
 * pages state.  Per batch row b and channel c (both dropped), t in [0,T):
 *
 *     wkv_t = ( sum_{i<t} e^{-(t-1-i) w + k_i} v_i  +  e^{u + k_t} v_t )
 *           / ( sum_{i<t} e^{-(t-1-i) w + k_i}      +  e^{u + k_t}     )
 *
 * w > 0 is the decay (passed in directly), u the bonus.  The most recent
 * past token (i = t-1) carries factor e^0: it is not decayed.
 *
 * Layout: k, v, y, gy, gk, gv are [B, T, C] row-major with C fastest;
 * w, u, gw, gu are [C].  Decode tensors are [L, B, C]; per-layer
 * parameters are [L, C].
 *
 * Every function here is pinned by tests under tests/ against values that
 * do not come from this file (closed forms, brute force finite differences,
 * limits, invariants); see tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define IDX(b, t, c) (((size_t)(b) * (size_t)T + (size_t)(t)) * (size_t)C + (size_t)(c))

int wkv_oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Forward, direct O(T^2) form: the definition above written out.  Each
 * exponent is formed first and exponentiated once. */
void wkv_oracle_forward_direct(int B, int T, int C, const double *w, const double *u,
                               const double *k, const double *v, double *y)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < C; ++c) {
            for (int t = 0; t < T; ++t) {
                double num = 0.0, den = 0.0;
                for (int i = 0; i < t; ++i) {
                    double e = exp(-(double)(t - 1 - i) * w[c] + k[IDX(b, i, c)]);
                    num += e * v[IDX(b, i, c)];
                    den += e;
                }
                double e = exp(u[c] + k[IDX(b, t, c)]);
                num += e * v[IDX(b, t, c)];
                den += e;
                y[IDX(b, t, c)] = num / den;
            }
        }
}

/* Forward, recurrent form ("eq. (8) can be written recursively").  Two
 * accumulators per channel: a_t = sum_{i<t} e^{-(t-1-i)w + k_i} v_i and
 * b_t likewise without v.  a_0 = b_0 = 0, and
 *     wkv_t   = (a_t + e^{u+k_t} v_t) / (b_t + e^{u+k_t})
 *     a_{t+1} = e^{-w} a_t + e^{k_t} v_t,   b_{t+1} = e^{-w} b_t + e^{k_t}.
 * No rescaling: in float64 the accumulators stay far from overflow for
 * |k| up to several hundred. */
void wkv_oracle_forward_recurrent(int B, int T, int C, const double *w, const double *u,
                                  const double *k, const double *v, double *y)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < C; ++c) {
            double a = 0.0, bb = 0.0;
            double decay = exp(-w[c]);
            for (int t = 0; t < T; ++t) {
                double kt = k[IDX(b, t, c)], vt = v[IDX(b, t, c)];
                double e = exp(u[c] + kt);
                y[IDX(b, t, c)] = (a + e * vt) / (bb + e);
                double ek = exp(kt);
                a = decay * a + ek * vt;
                bb = decay * bb + ek;
            }
        }
}

/* Forward from a carried state: the same operator over T more tokens of a
 * sequence whose earlier tokens are summarised by the state (num, den, pp)
 * [B, C] in the convention of wkv_oracle_state (a = num e^{pp} and
 * b = den e^{pp} are the sums a_0, b_0 over the earlier tokens; pp = -1e38
 * with num = den = 0 is the empty state).  The earlier tokens decay with
 * the distance like any others, so for t in [0, T):
 *     a_t = e^{-t w} a_0 + sum_{i<t} e^{-(t-1-i) w + k_i} v_i  (b_t alike)
 *     wkv_t = (a_t + e^{u+k_t} v_t) / (b_t + e^{u+k_t}).
 * Evaluated by the recurrence of wkv_oracle_forward_recurrent with the sums
 * kept as (A, Bs, M), a = A e^{M}, so that a state with a large pp does not
 * overflow a double; M is the running maximum of the exponents.  num_in
 * (with den_in, pp_in) may be NULL: the empty state.  The state after the
 * T tokens is written to num_out, den_out, pp_out ([B, C], may be NULL) in
 * the same convention. */
void wkv_oracle_forward_state(int B, int T, int C, const double *w, const double *u,
                              const double *k, const double *v, const double *num_in,
                              const double *den_in, const double *pp_in, double *y,
                              double *num_out, double *den_out, double *pp_out)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < C; ++c) {
            size_t o = (size_t)b * (size_t)C + (size_t)c;
            double A = 0.0, Bs = 0.0, M = -INFINITY;
            if (num_in && pp_in[o] > -1e37) {
                A = num_in[o];
                Bs = den_in[o];
                M = pp_in[o];
            }
            for (int t = 0; t < T; ++t) {
                double kt = k[IDX(b, t, c)], vt = v[IDX(b, t, c)];
                double ek = u[c] + kt;                 /* exponent of the current token's weight */
                double q = M > ek ? M : ek;
                double sp = exp(M - q), sc = exp(ek - q);
                y[IDX(b, t, c)] = (A * sp + vt * sc) / (Bs * sp + sc);
                double m2 = (M - w[c]) > kt ? (M - w[c]) : kt;
                double dp = exp(M - w[c] - m2), dk = exp(kt - m2);
                A = A * dp + vt * dk;
                Bs = Bs * dp + dk;
                M = m2;
            }
            if (num_out) {
                int seen = M > -INFINITY;
                num_out[o] = seen ? A : 0.0;
                den_out[o] = seen ? Bs : 0.0;
                pp_out[o] = seen ? M : -1e38;
            }
        }
}

/* Backward, reverse-mode differentiation of the recurrent form.  Given the
 * upstream gradient gy = dLoss/dwkv, returns gk, gv ([B,T,C]) and gw, gu
 * ([C], summed over b and t).  With N_t, D_t the numerator and denominator
 * of wkv_t, e_t = e^{u+k_t}, gN_t = gy_t / D_t and gD_t = -gy_t wkv_t / D_t,
 * and adjoints la_t = dLoss/da_t, lb_t = dLoss/db_t (la_T = lb_T = 0):
 *     gk_t = (gN_t v_t + gD_t) e_t + (la_{t+1} v_t + lb_{t+1}) e^{k_t}
 *     gv_t = gN_t e_t + la_{t+1} e^{k_t}
 *     gu  += (gN_t v_t + gD_t) e_t
 *     gw  += -e^{-w} (la_{t+1} a_t + lb_{t+1} b_t)
 *     la_t = gN_t + e^{-w} la_{t+1},    lb_t = gD_t + e^{-w} lb_{t+1}.
 * The forward accumulators are kept per step (O(T) memory per channel). */
void wkv_oracle_backward_adjoint(int B, int T, int C, const double *w, const double *u,
                                 const double *k, const double *v, const double *gy,
                                 double *gw, double *gu, double *gk, double *gv)
{
    /* per-(b, c) partial sums of gw, gu, reduced over b in a fixed order
     * afterwards so the result does not depend on the thread count */
    double *pw = (double *)malloc(sizeof(double) * (size_t)B * (size_t)C);
    double *pu = (double *)malloc(sizeof(double) * (size_t)B * (size_t)C);
#pragma omp parallel
    {
        /* per-thread storage of the forward accumulators a_t, b_t */
        double *a = (double *)malloc(sizeof(double) * (size_t)(T + 1));
        double *bb = (double *)malloc(sizeof(double) * (size_t)(T + 1));
#pragma omp for collapse(2) schedule(static)
        for (int b = 0; b < B; ++b)
            for (int c = 0; c < C; ++c) {
                double decay = exp(-w[c]);
                a[0] = 0.0;
                bb[0] = 0.0;
                for (int t = 0; t < T; ++t) {
                    double ek = exp(k[IDX(b, t, c)]);
                    a[t + 1] = decay * a[t] + ek * v[IDX(b, t, c)];
                    bb[t + 1] = decay * bb[t] + ek;
                }
                double la = 0.0, lb = 0.0, sgw = 0.0, sgu = 0.0;
                for (int t = T - 1; t >= 0; --t) {
                    double kt = k[IDX(b, t, c)], vt = v[IDX(b, t, c)], g = gy[IDX(b, t, c)];
                    double e = exp(u[c] + kt), ek = exp(kt);
                    double D = bb[t] + e;
                    double N = a[t] + e * vt;
                    double yt = N / D;
                    double gN = g / D;
                    double gD = -g * yt / D;
                    gk[IDX(b, t, c)] = (gN * vt + gD) * e + (la * vt + lb) * ek;
                    gv[IDX(b, t, c)] = gN * e + la * ek;
                    sgu += (gN * vt + gD) * e;
                    sgw += -decay * (la * a[t] + lb * bb[t]);
                    la = gN + decay * la;
                    lb = gD + decay * lb;
                }
                pw[(size_t)b * (size_t)C + (size_t)c] = sgw;
                pu[(size_t)b * (size_t)C + (size_t)c] = sgu;
            }
        free(a);
        free(bb);
    }
    for (int c = 0; c < C; ++c) {
        double sw = 0.0, su = 0.0;
        for (int b = 0; b < B; ++b) {
            sw += pw[(size_t)b * (size_t)C + (size_t)c];
            su += pu[(size_t)b * (size_t)C + (size_t)c];
        }
        gw[c] = sw;
        gu[c] = su;
    }
    free(pw);
    free(pu);
}

/* Backward pass of a segment that starts from a given state and whose end
 * sums feed later tokens: the gradient with respect to a carried state, and
 * the piece a sequence split along time needs per segment.  The segment's
 * sums start at a_0 = num_in e^{pp_in}, b_0 = den_in e^{pp_in} (zero for a
 * NULL or empty state) and the loss is
 *     L = sum_t gy_t wkv_t + ga_end a_T + gb_end b_T,
 * ga_end, gb_end [B, C] the gradient reaching the end sums from the tokens
 * after the segment (NULL: none).  The recurrence of
 * wkv_oracle_backward_adjoint, started from la_T = ga_end, lb_T = gb_end,
 * gives gw (the start state's decay through the segment included), gu, gk,
 * gv, and the adjoint of the start sums ga_start = la_0 = dL/da_0,
 * gb_start = lb_0 ([B, C]; NULL: not returned).  Unscaled sums: moderate k
 * only. */
void wkv_oracle_backward_state(int B, int T, int C, const double *w, const double *u, const double *k,
                               const double *v, const double *gy, const double *num_in,
                               const double *den_in, const double *pp_in, const double *ga_end,
                               const double *gb_end, double *gw, double *gu, double *gk, double *gv,
                               double *ga_start, double *gb_start)
{
    double *a = (double *)malloc(sizeof(double) * (size_t)(T + 1));
    double *bb = (double *)malloc(sizeof(double) * (size_t)(T + 1));
    double *pw = (double *)malloc(sizeof(double) * (size_t)B * (size_t)C);
    double *pu = (double *)malloc(sizeof(double) * (size_t)B * (size_t)C);
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < C; ++c) {
            size_t o = (size_t)b * (size_t)C + (size_t)c;
            double decay = exp(-w[c]);
            int given = num_in && pp_in[o] > -1e37;
            a[0] = given ? num_in[o] * exp(pp_in[o]) : 0.0;
            bb[0] = given ? den_in[o] * exp(pp_in[o]) : 0.0;
            for (int t = 0; t < T; ++t) {
                double ek = exp(k[IDX(b, t, c)]);
                a[t + 1] = decay * a[t] + ek * v[IDX(b, t, c)];
                bb[t + 1] = decay * bb[t] + ek;
            }
            double la = ga_end ? ga_end[o] : 0.0, lb = gb_end ? gb_end[o] : 0.0, sgw = 0.0, sgu = 0.0;
            for (int t = T - 1; t >= 0; --t) {
                double kt = k[IDX(b, t, c)], vt = v[IDX(b, t, c)], g = gy[IDX(b, t, c)];
                double e = exp(u[c] + kt), ek = exp(kt);
                double D = bb[t] + e;
                double yt = (a[t] + e * vt) / D;
                double gN = g / D;
                double gD = -g * yt / D;
                gk[IDX(b, t, c)] = (gN * vt + gD) * e + (la * vt + lb) * ek;
                gv[IDX(b, t, c)] = gN * e + la * ek;
                sgu += (gN * vt + gD) * e;
                sgw += -decay * (la * a[t] + lb * bb[t]);
                la = gN + decay * la;
                lb = gD + decay * lb;
            }
            pw[o] = sgw;
            pu[o] = sgu;
            if (ga_start) ga_start[o] = la;
            if (gb_start) gb_start[o] = lb;
        }
    for (int c = 0; c < C; ++c) {
        double sw = 0.0, su = 0.0;
        for (int b = 0; b < B; ++b) {
            sw += pw[(size_t)b * (size_t)C + (size_t)c];
            su += pu[(size_t)b * (size_t)C + (size_t)c];
        }
        gw[c] = sw;
        gu[c] = su;
    }
    free(a);
    free(bb);
    free(pw);
    free(pu);
}

/* Backward, direct O(T^2) derivative of the definition.  For i < t the
 * weight of token i in wkv_t is W_ti = e^{-(t-1-i)w + k_i}; for i = t it is
 * e^{u+k_t}.  Then, with D_t the denominator:
 *     d wkv_t / d v_i = W_ti / D_t
 *     d wkv_t / d k_i = W_ti (v_i - wkv_t) / D_t
 *     d wkv_t / d u   = e^{u+k_t} (v_t - wkv_t) / D_t
 *     d wkv_t / d w   = -sum_{i<t} (t-1-i) W_ti (v_i - wkv_t) / D_t
 * and each is contracted with gy_t.  Shares nothing with the adjoint form. */
void wkv_oracle_backward_direct(int B, int T, int C, const double *w, const double *u,
                                const double *k, const double *v, const double *gy,
                                double *gw, double *gu, double *gk, double *gv)
{
    for (int c = 0; c < C; ++c) {
        gw[c] = 0.0;
        gu[c] = 0.0;
    }
    for (size_t n = 0; n < (size_t)B * (size_t)T * (size_t)C; ++n) {
        gk[n] = 0.0;
        gv[n] = 0.0;
    }
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; ++c)
        for (int b = 0; b < B; ++b)
            for (int t = 0; t < T; ++t) {
                double D = 0.0, N = 0.0;
                for (int i = 0; i < t; ++i) {
                    double W = exp(-(double)(t - 1 - i) * w[c] + k[IDX(b, i, c)]);
                    D += W;
                    N += W * v[IDX(b, i, c)];
                }
                double Wt = exp(u[c] + k[IDX(b, t, c)]);
                D += Wt;
                N += Wt * v[IDX(b, t, c)];
                double yt = N / D, g = gy[IDX(b, t, c)];
                for (int i = 0; i < t; ++i) {
                    double W = exp(-(double)(t - 1 - i) * w[c] + k[IDX(b, i, c)]);
                    double vi = v[IDX(b, i, c)];
                    gv[IDX(b, i, c)] += g * W / D;
                    gk[IDX(b, i, c)] += g * W * (vi - yt) / D;
                    gw[c] += -g * (double)(t - 1 - i) * W * (vi - yt) / D;
                }
                double vt = v[IDX(b, t, c)];
                gv[IDX(b, t, c)] += g * Wt / D;
                gk[IDX(b, t, c)] += g * Wt * (vt - yt) / D;
                gu[c] += g * Wt * (vt - yt) / D;
            }
}

/* The carried state after the first t tokens (t in [0, T]) in the
 * (num, den, pp) convention of the decode step: a_t = num * e^{pp},
 * b_t = den * e^{pp}, where pp is the exact running maximum of the
 * exponents, pp_t = max_{i<t} (k_i - (t-1-i) w), and pp_0 = -1e38 with
 * num = den = 0 (no token seen).  Written from the definition (direct sum),
 * not from a recurrence.  Outputs are [B, C]. */
void wkv_oracle_state(int B, int T, int C, const double *w, const double *k, const double *v,
                      int t, double *num, double *den, double *pp)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < C; ++c) {
            size_t o = (size_t)b * (size_t)C + (size_t)c;
            if (t <= 0) {
                num[o] = 0.0;
                den[o] = 0.0;
                pp[o] = -1e38;
                continue;
            }
            double m = -INFINITY;
            for (int i = 0; i < t; ++i) {
                double ex = k[IDX(b, i, c)] - (double)(t - 1 - i) * w[c];
                if (ex > m) m = ex;
            }
            double sa = 0.0, sb = 0.0;
            for (int i = 0; i < t; ++i) {
                double W = exp(k[IDX(b, i, c)] - (double)(t - 1 - i) * w[c] - m);
                sa += W * v[IDX(b, i, c)];
                sb += W;
            }
            num[o] = sa;
            den[o] = sb;
            pp[o] = m;
        }
}

/* One decode step of L independent time-mixing layers (RNN mode).  Per
 * (l, b, c), with per-layer parameters indexed (l, c):
 *   token shift, eq. (7):  xk = mu_k x + (1 - mu_k) x_prev  (xv, xr alike)
 *   wkv from the carried state and this token's k, v:
 *        a = num e^{pp}, b = den e^{pp},
 *        wkv = (a + e^{u+k} v) / (b + e^{u+k})
 *   gate, eq. (9):  y = sigmoid(r) * wkv = wkv / (1 + e^{-r})
 *   state update:   a' = e^{-w} a + e^{k} v,  b' = e^{-w} b + e^{k},
 *                   pp' = max(pp - w, k),  num' = a' e^{-pp'},  den' = b' e^{-pp'}.
 * num, den, pp are updated in place.  xk, xv, xr may be NULL. */
void wkv_oracle_decode_step(int L, int B, int C, const double *x, const double *x_prev,
                            const double *mu_k, const double *mu_v, const double *mu_r,
                            const double *r, const double *k, const double *v,
                            const double *w, const double *u, double *num, double *den,
                            double *pp, double *y, double *xk, double *xv, double *xr)
{
#pragma omp parallel for collapse(3) schedule(static)
    for (int l = 0; l < L; ++l)
        for (int b = 0; b < B; ++b)
            for (int c = 0; c < C; ++c) {
                size_t o = ((size_t)l * (size_t)B + (size_t)b) * (size_t)C + (size_t)c;
                size_t p = (size_t)l * (size_t)C + (size_t)c;
                if (xk) xk[o] = mu_k[p] * x[o] + (1.0 - mu_k[p]) * x_prev[o];
                if (xv) xv[o] = mu_v[p] * x[o] + (1.0 - mu_v[p]) * x_prev[o];
                if (xr) xr[o] = mu_r[p] * x[o] + (1.0 - mu_r[p]) * x_prev[o];
                double scale = exp(pp[o]);
                double a = num[o] * scale, bb = den[o] * scale;
                double e = exp(u[p] + k[o]);
                double wkv = (a + e * v[o]) / (bb + e);
                y[o] = wkv / (1.0 + exp(-r[o]));
                double ek = exp(k[o]);
                double a2 = exp(-w[p]) * a + ek * v[o];
                double b2 = exp(-w[p]) * bb + ek;
                double pp2 = pp[o] - w[p] > k[o] ? pp[o] - w[p] : k[o];
                num[o] = a2 * exp(-pp2);
                den[o] = b2 * exp(-pp2);
                pp[o] = pp2;
            }
}

/* The time-mixing output with its receptance gate, eq. (9) of "RWKV解读"
 * section "3、RWKV的网络架构" (the wkv result is multiplied elementwise by
 * sigmoid of the receptance r before the output projection): per (b, t, c)
 *     out_t = sigmoid(r_t) wkv_t,   sigmoid(r) = 1 / (1 + e^{-r}),
 * with wkv_t the direct sum of wkv_oracle_forward_direct.  r is [B, T, C]. */
void wkv_oracle_forward_gated(int B, int T, int C, const double *w, const double *u, const double *k,
                              const double *v, const double *r, double *out)
{
    wkv_oracle_forward_direct(B, T, C, w, u, k, v, out);
    size_t n = (size_t)B * (size_t)T * (size_t)C;
    for (size_t i = 0; i < n; ++i)
        out[i] = out[i] / (1.0 + exp(-r[i]));
}

/* The same gated output through the recurrent form: sigmoid(r_t) times
 * wkv_t of wkv_oracle_forward_recurrent.  O(T) per channel, so it is the
 * form the CPU timing uses; it equals wkv_oracle_forward_gated (the direct
 * O(T^2) sums) up to rounding. */
void wkv_oracle_forward_gated_recurrent(int B, int T, int C, const double *w, const double *u, const double *k,
                                        const double *v, const double *r, double *out)
{
    wkv_oracle_forward_recurrent(B, T, C, w, u, k, v, out);
    size_t n = (size_t)B * (size_t)T * (size_t)C;
    for (size_t i = 0; i < n; ++i)
        out[i] = out[i] / (1.0 + exp(-r[i]));
}

/* Gradients of sum(gout * out) for the gated output above.  wkv_t reaches
 * the loss only through out_t, with factor sigmoid(r_t), so the gradient
 * that enters the recurrence's reverse mode is gy_t = gout_t sigmoid(r_t)
 * (giving gw, gu, gk, gv as wkv_oracle_backward_adjoint); and, from the
 * derivative sigmoid'(r) = sigmoid(r) (1 - sigmoid(r)),
 *     gr_t = gout_t wkv_t sigmoid(r_t) (1 - sigmoid(r_t)).
 * wkv_t here comes from the recurrent form (wkv_oracle_forward_recurrent). */
void wkv_oracle_backward_gated(int B, int T, int C, const double *w, const double *u, const double *k,
                               const double *v, const double *r, const double *gout, double *gw,
                               double *gu, double *gk, double *gv, double *gr)
{
    size_t n = (size_t)B * (size_t)T * (size_t)C;
    double *y = (double *)malloc(sizeof(double) * n);
    double *gy = (double *)malloc(sizeof(double) * n);
    wkv_oracle_forward_recurrent(B, T, C, w, u, k, v, y);
    for (size_t i = 0; i < n; ++i) {
        double s = 1.0 / (1.0 + exp(-r[i]));
        gy[i] = gout[i] * s;
        gr[i] = gout[i] * y[i] * s * (1.0 - s);
    }
    wkv_oracle_backward_adjoint(B, T, C, w, u, k, v, gy, gw, gu, gk, gv);
    free(y);
    free(gy);
}

/* The state after consecutive segments of one sequence, from each segment's
 * own state (after its tokens, from the empty state) and its length: the
 * prefix combination that lets segments of one long sequence run apart
 * ("RWKV解读" section "3、RWKV的网络架构": eq. (8) written recursively; qiita
 * "Trainingについて": the decay does not depend on the data, so a segment's
 * effect on the carried state is "decay by its length, add its own sums").
 * In the decode step's convention a = num e^{pp}, b = den e^{pp}; a token
 * decays once for every later token, so after a state P and a segment of n
 * tokens with own sums a_S, b_S:
 *     a = e^{-n w} a_P + a_S,   b = e^{-n w} b_P + b_S,
 * kept at the scale of the larger exponent.  states is [n][3][B][C] (planes
 * num, den, pp; pp <= -1e37 marks an empty segment), lengths [n], out
 * [3][B][C] (the empty state, num = den = 0 and pp = -1e38, if no segment
 * has a token). */
void wkv_oracle_state_fold(int B, int C, const double *w, int n, const double *states,
                           const long long *lengths, double *out)
{
    size_t bc = (size_t)B * (size_t)C;
    for (size_t o = 0; o < bc; ++o) {
        int c = (int)(o % (size_t)C);
        double A = 0.0, Bs = 0.0, M = -INFINITY;
        for (int i = 0; i < n; ++i) {
            const double *st = states + (size_t)i * 3 * bc;
            double Md = M - (double)lengths[i] * w[c];
            if (st[2 * bc + o] <= -1e37) {
                M = Md;
                continue;
            }
            double m2 = Md > st[2 * bc + o] ? Md : st[2 * bc + o];
            double dp = exp(Md - m2), ds = exp(st[2 * bc + o] - m2);
            A = A * dp + st[o] * ds;
            Bs = Bs * dp + st[bc + o] * ds;
            M = m2;
        }
        int seen = M > -INFINITY;
        out[o] = seen ? A : 0.0;
        out[bc + o] = seen ? Bs : 0.0;
        out[2 * bc + o] = seen ? M : -1e38;
    }
}

/* The pointwise parts of channel mixing (segmentfault "RWKV解读" section
 * "3、RWKV的网络架构", eq. (10), whose body the page lost; qiita "RWKV
 * についての調査記録": channel mixing computes K, then V from it, then gates
 * with a sigmoid; "Инновационная архитектура RWKV", section "Механизмы
 * взаимодействия": the projected signal goes through a squared ReLU and is
 * multiplied by a sigmoid forget gate).  Read here as: between the key and
 * value projections
 *     a = max(k, 0)^2,          backward  gk = 2 max(k, 0) ga,
 * and after the value projection vk = W_v a, with r the receptance,
 *     out = sigmoid(r) vk,      backward  gvk = gout sigmoid(r),
 *                                         gr  = gout vk sigmoid(r) (1 - sigmoid(r)).
 * Elementwise over n values. */
void wkv_oracle_sqrelu(size_t n, const double *k, double *a)
{
    for (size_t i = 0; i < n; ++i) {
        double p = k[i] > 0.0 ? k[i] : 0.0;
        a[i] = p * p;
    }
}

void wkv_oracle_sqrelu_backward(size_t n, const double *k, const double *ga, double *gk)
{
    for (size_t i = 0; i < n; ++i)
        gk[i] = 2.0 * (k[i] > 0.0 ? k[i] : 0.0) * ga[i];
}

void wkv_oracle_cmix_gate(size_t n, const double *r, const double *vk, double *out)
{
    for (size_t i = 0; i < n; ++i)
        out[i] = vk[i] / (1.0 + exp(-r[i]));
}

void wkv_oracle_cmix_gate_backward(size_t n, const double *r, const double *vk, const double *gout,
                                   double *gr, double *gvk)
{
    for (size_t i = 0; i < n; ++i) {
        double s = 1.0 / (1.0 + exp(-r[i]));
        gvk[i] = gout[i] * s;
        gr[i] = gout[i] * vk[i] * s * (1.0 - s);
    }
}

/* Token shift of the training path, eq. (7) of "RWKV解读" section
 * "3、RWKV的网络架构" (the input of each projection is a weighted sum of the
 * current and the previous token; segmentfault and "Инновационная
 * архитектура RWKV", "Механизмы взаимодействия"): per (b, t, c), with
 * x_{-1} = x0 (the last token before the sequence, [B, C]; NULL: zeros),
 *     xk_t = mu_k x_t + (1 - mu_k) x_{t-1}   (xv, xr with mu_v, mu_r).
 * Backward, given gxk, gxv, gxr [B, T, C]: each x_t feeds its own mixes
 * with weight mu and the next token's with weight 1 - mu, so
 *     gx_t  = sum_m mu_m gxm_t + (1 - mu_m) gxm_{t+1}   (no t+1 term at T-1)
 *     gx0   = sum_m (1 - mu_m) gxm_0                    ([B, C], may be NULL)
 *     gmu_m = sum_{b,t} gxm_t (x_t - x_{t-1})           ([C]). */
void wkv_oracle_token_shift(int B, int T, int C, const double *x, const double *x0, const double *mu_k,
                            const double *mu_v, const double *mu_r, double *xk, double *xv, double *xr)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int b = 0; b < B; ++b)
        for (int c = 0; c < C; ++c)
            for (int t = 0; t < T; ++t) {
                double cur = x[IDX(b, t, c)];
                double prev = t > 0 ? x[IDX(b, t - 1, c)] : (x0 ? x0[(size_t)b * C + c] : 0.0);
                xk[IDX(b, t, c)] = mu_k[c] * cur + (1.0 - mu_k[c]) * prev;
                xv[IDX(b, t, c)] = mu_v[c] * cur + (1.0 - mu_v[c]) * prev;
                xr[IDX(b, t, c)] = mu_r[c] * cur + (1.0 - mu_r[c]) * prev;
            }
}

void wkv_oracle_token_shift_backward(int B, int T, int C, const double *x, const double *x0,
                                     const double *mu_k, const double *mu_v, const double *mu_r,
                                     const double *gxk, const double *gxv, const double *gxr, double *gx,
                                     double *gx0, double *gmu_k, double *gmu_v, double *gmu_r)
{
#pragma omp parallel for schedule(static)
    for (int c = 0; c < C; ++c) {
        double sk = 0.0, sv = 0.0, sr = 0.0;
        for (int b = 0; b < B; ++b)
            for (int t = 0; t < T; ++t) {
                size_t i = IDX(b, t, c);
                double g = mu_k[c] * gxk[i] + mu_v[c] * gxv[i] + mu_r[c] * gxr[i];
                if (t + 1 < T) {
                    size_t n = IDX(b, t + 1, c);
                    g += (1.0 - mu_k[c]) * gxk[n] + (1.0 - mu_v[c]) * gxv[n] + (1.0 - mu_r[c]) * gxr[n];
                }
                gx[i] = g;
                double prev = t > 0 ? x[IDX(b, t - 1, c)] : (x0 ? x0[(size_t)b * C + c] : 0.0);
                double d = x[i] - prev;
                sk += gxk[i] * d;
                sv += gxv[i] * d;
                sr += gxr[i] * d;
            }
        gmu_k[c] = sk;
        gmu_v[c] = sv;
        gmu_r[c] = sr;
        if (gx0)
            for (int b = 0; b < B; ++b) {
                size_t i = IDX(b, 0, c);
                gx0[(size_t)b * C + c] = (1.0 - mu_k[c]) * gxk[i] + (1.0 - mu_v[c]) * gxv[i] + (1.0 - mu_r[c]) * gxr[i];
            }
    }
}
