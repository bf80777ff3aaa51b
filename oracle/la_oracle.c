/*
 * la_oracle.c -- the oracle for causal linear attention, retention and gated
 * linear attention: the plain recurrent form, evaluated in fp64.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may link, load or call
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline
 * leg do. It shares no code, header, table or constant generator with the CUDA
 * library.
 *
 * What it computes, for every (b, h) sequence independently:
 *
 *   S_0 = 0 (d_k x d_v), z_0 = 0 (d_k)          "causal linear attention as an
 *                                                 RNN": S_0 = Z_0 = 0
 *   for t = 0 .. L-1:
 *     qf = phi(q_t), kf = phi(k_t)               phi = identity or elu(x)+1
 *                                                 (learnllm m22, "The Math:
 *                                                 Linear Attention")
 *     a  = 1 | gamma_h | alpha_t                 the gate A_t of the unified
 *                                                 recurrence (learnllm m22,
 *                                                 "Interactive Exploration")
 *     S  = diag(a) S + kf v_t^T                  k v^T orientation, d_k x d_v
 *                                                 (insideout lesson 16, Ex. 1.1)
 *     z  = a * z + kf                            only when normalised
 *     out_t = qf^T S            (unnormalised)   read AFTER the update
 *     out_t = qf^T S / (qf . z) (normalised)     (linear_sparse_attention.py,
 *                                                 linear_attn_recurrent)
 *
 * alpha_t[i] = exp(logsigmoid(g_t[i]) / 16) for the per-channel gate (the gated
 * linear attention gate with temperature 16; Yang et al. 2023, cited on the
 * troisinh and learnllm pages). logsigmoid is evaluated in the overflow-free
 * split form. The denominator has no epsilon: phi > 0 keeps it positive
 * (learnllm m22, "Common Pitfalls" 1).
 *
 * Inputs arrive as float32 arrays: bf16 inputs are carried exactly in float32,
 * and every value is upcast to double before any arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* mode bits: the problem statement's flags, restated here for the oracle */
#define OR_PHI_ELU1     0x1
#define OR_NORMALIZE    0x2
#define OR_GATE_HEAD    0x4
#define OR_GATE_CHANNEL 0x8

static double or_phi(double x, int elu1)
{
    if (!elu1) return x;
    return x > 0.0 ? x + 1.0 : exp(x);   /* elu with alpha = 1, plus one */
}

static double or_log_sigmoid(double x)
{
    /* log(1/(1+e^-x)), split so that neither branch overflows */
    if (x >= 0.0) return -log1p(exp(-x));
    return x - log1p(exp(x));
}

/* One sequence of L tokens; S (dk*dv) and z (dk) hold the running state on
 * entry and on exit. g is [L, dk] for the per-channel gate, else unused. */
static void or_sequence(const float *q, const float *k, const float *v,
                        const float *g, double gamma, int L, int dk, int dv,
                        int mode, double *S, double *z, double *out)
{
    const int elu1 = (mode & OR_PHI_ELU1) != 0;
    const int norm = (mode & OR_NORMALIZE) != 0;
    double *qf = (double *)malloc(sizeof(double) * (size_t)dk * 3);
    double *kf = qf + dk;
    double *a = kf + dk;
    for (int t = 0; t < L; ++t) {
        const float *qt = q + (size_t)t * dk;
        const float *kt = k + (size_t)t * dk;
        const float *vt = v + (size_t)t * dv;
        for (int i = 0; i < dk; ++i) {
            qf[i] = or_phi((double)qt[i], elu1);
            kf[i] = or_phi((double)kt[i], elu1);
            if (mode & OR_GATE_CHANNEL)
                a[i] = exp(or_log_sigmoid((double)g[(size_t)t * dk + i]) / 16.0);
            else if (mode & OR_GATE_HEAD)
                a[i] = gamma;
            else
                a[i] = 1.0;
        }
        for (int i = 0; i < dk; ++i) {
            double *Si = S + (size_t)i * dv;
            for (int j = 0; j < dv; ++j)
                Si[j] = a[i] * Si[j] + kf[i] * (double)vt[j];
            if (norm) z[i] = a[i] * z[i] + kf[i];
        }
        double den = 0.0;
        if (norm)
            for (int i = 0; i < dk; ++i) den += qf[i] * z[i];
        double *ot = out + (size_t)t * dv;
        for (int j = 0; j < dv; ++j) {
            double num = 0.0;
            for (int i = 0; i < dk; ++i) num += qf[i] * S[(size_t)i * dv + j];
            ot[j] = norm ? num / den : num;
        }
    }
    free(qf);
}

/*
 * oracle_forward: the whole forward pass over q, k, v [B,H,L,dk|dv].
 *   gate: NULL, gamma[H] (OR_GATE_HEAD) or g[B,H,L,dk] (OR_GATE_CHANNEL)
 *   state_in: NULL (start from zero) or [B,H] blocks of S (dk*dv) followed,
 *             when normalised, by z (dk) -- the block layout of state_out
 *   out: [B,H,L,dv] doubles; state_out: same block layout as state_in
 * Returns 0, or -1 on a bad argument.
 */
int oracle_forward(const float *q, const float *k, const float *v,
                   const float *gate, const double *state_in, int B, int H,
                   int L, int dk, int dv, int mode, double *out,
                   double *state_out, int nthreads)
{
    if (B < 0 || H < 0 || L < 0 || dk <= 0 || dv <= 0) return -1;
    if ((mode & OR_GATE_HEAD) && (mode & OR_GATE_CHANNEL)) return -1;
    if ((mode & (OR_GATE_HEAD | OR_GATE_CHANNEL)) && !gate) return -1;
    const int norm = (mode & OR_NORMALIZE) != 0;
    const size_t blk = (size_t)dk * dv + (norm ? (size_t)dk : 0);
    const long nbh = (long)B * H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long bh = 0; bh < nbh; ++bh) {
        const int h = (int)(bh % H);
        double *st = state_out + (size_t)bh * blk;
        if (state_in) memcpy(st, state_in + (size_t)bh * blk, blk * sizeof(double));
        else memset(st, 0, blk * sizeof(double));
        const float *g = NULL;
        double gamma = 1.0;
        if (mode & OR_GATE_CHANNEL) g = gate + (size_t)bh * L * dk;
        if (mode & OR_GATE_HEAD) gamma = (double)gate[h];
        or_sequence(q + (size_t)bh * L * dk, k + (size_t)bh * L * dk,
                    v + (size_t)bh * L * dv, g, gamma, L, dk, dv, mode, st,
                    norm ? st + (size_t)dk * dv : NULL, out + (size_t)bh * L * dv);
    }
    (void)nthreads;
    return 0;
}

/* oracle_decode_step: one token per (b, h) on an existing state, in place.
 * q, k: [B,H,dk]; v: [B,H,dv]; gate as above with L = 1; state: block layout
 * as above; out: [B,H,dv]. It is oracle_forward at L = 1 from state. */
int oracle_decode_step(const float *q, const float *k, const float *v,
                       const float *gate, double *state, int B, int H, int dk,
                       int dv, int mode, double *out, int nthreads)
{
    if (B < 0 || H < 0 || dk <= 0 || dv <= 0) return -1;
    if ((mode & OR_GATE_HEAD) && (mode & OR_GATE_CHANNEL)) return -1;
    if ((mode & (OR_GATE_HEAD | OR_GATE_CHANNEL)) && !gate) return -1;
    const int norm = (mode & OR_NORMALIZE) != 0;
    const size_t blk = (size_t)dk * dv + (norm ? (size_t)dk : 0);
    const long nbh = (long)B * H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(static) num_threads(nthreads)
#endif
    for (long bh = 0; bh < nbh; ++bh) {
        const int h = (int)(bh % H);
        double *st = state + (size_t)bh * blk;
        const float *g = NULL;
        double gamma = 1.0;
        if (mode & OR_GATE_CHANNEL) g = gate + (size_t)bh * dk;
        if (mode & OR_GATE_HEAD) gamma = (double)gate[h];
        or_sequence(q + (size_t)bh * dk, k + (size_t)bh * dk, v + (size_t)bh * dv,
                    g, gamma, 1, dk, dv, mode, st, norm ? st + (size_t)dk * dv : NULL,
                    out + (size_t)bh * dv);
    }
    (void)nthreads;
    return 0;
}

/*
 * oracle_delta_forward: the delta rule (DeltaNet), recurrent, fp64
 * (linear_sparse_attention.py, "delta_rule_recurrent"). The state is d_v x d_k,
 * the v k^T orientation of that function; per token, in the page's two steps:
 *     S = S (I - beta_t k_t k_t^T)      erase what S returns for k_t
 *     S = S + beta_t v_t k_t^T          write v_t in its place
 *     out_t = S q_t                     read AFTER the update (the reading of
 *                                       the other forms; the page returns states)
 * k_t is taken as given (the page assumes unit-norm keys and leaves the
 * normalisation to the caller).
 *   q, k: [B,H,L,dk]; v: [B,H,L,dv]; beta: [B,H,L]
 *   state_in: NULL (start from zero) or [B,H] blocks of dv*dk (row i = value
 *             dimension i); out: [B,H,L,dv]; state_out: same blocks as state_in
 * Returns 0, or -1 on a bad argument.
 */
int oracle_delta_forward(const float *q, const float *k, const float *v,
                         const float *beta, const double *state_in, int B, int H,
                         int L, int dk, int dv, double *out, double *state_out,
                         int nthreads)
{
    if (B < 0 || H < 0 || L < 0 || dk <= 0 || dv <= 0 || !beta) return -1;
    const size_t blk = (size_t)dv * dk;
    const long nbh = (long)B * H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long bh = 0; bh < nbh; ++bh) {
        double *S = state_out + (size_t)bh * blk;
        if (state_in) memcpy(S, state_in + (size_t)bh * blk, blk * sizeof(double));
        else memset(S, 0, blk * sizeof(double));
        double *kt = (double *)malloc(sizeof(double) * ((size_t)dk * 2 + dv));
        double *qt = kt + dk;
        double *Sk = qt + dk;
        for (int t = 0; t < L; ++t) {
            const size_t tk = ((size_t)bh * L + t) * dk, tv = ((size_t)bh * L + t) * dv;
            const double b = (double)beta[(size_t)bh * L + t];
            for (int j = 0; j < dk; ++j) {
                kt[j] = (double)k[tk + j];
                qt[j] = (double)q[tk + j];
            }
            /* S (I - b k k^T) = S - b (S k) k^T */
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * kt[j];
                Sk[i] = acc;
            }
            for (int i = 0; i < dv; ++i)
                for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] -= b * Sk[i] * kt[j];
            /* + b v k^T */
            for (int i = 0; i < dv; ++i) {
                const double vi = (double)v[tv + i];
                for (int j = 0; j < dk; ++j) S[(size_t)i * dk + j] += b * vi * kt[j];
            }
            double *ot = out + tv;
            for (int i = 0; i < dv; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dk; ++j) acc += S[(size_t)i * dk + j] * qt[j];
                ot[i] = acc;
            }
        }
        free(kt);
    }
    (void)nthreads;
    return 0;
}

/*
 * oracle_group_norm_swish: the RetNet output epilogue, fp64 (learnllm m22,
 * "Retention": retention keeps no normaliser; RetNet steadies its output with
 * a GroupNorm and a swish gate instead). One group per head, so every
 * (b, h, t) row of dv outputs is normalised on its own:
 *     mean = sum_i x_i / dv,   var = sum_i (x_i - mean)^2 / dv   (biased)
 *     y_i  = (x_i - mean) / sqrt(var + eps) * weight[h][i] + bias[h][i]
 *     out_i = swish(og_i) * y_i,   swish(u) = u sigmoid(u) = u / (1 + e^-u)
 * og is the output gate (the caller's projection of the layer input); the
 * output projection that follows is the caller's too.
 *   x, out: [B,H,L,dv] fp64 (out may be x); og: [B,H,L,dv];
 *   weight, bias: [H][dv], or NULL for 1 and 0
 * Returns 0, or -1 on a bad argument.
 */
static double or_swish(double u)
{
    /* u / (1 + e^-u), written so that neither tail overflows */
    if (u >= 0.0) return u / (1.0 + exp(-u));
    const double e = exp(u);
    return u * e / (1.0 + e);
}

int oracle_group_norm_swish(const double *x, const float *og, const float *weight,
                            const float *bias, double eps, int B, int H, int L, int dv,
                            double *out)
{
    if (B < 0 || H < 0 || L < 0 || dv <= 0 || !(eps >= 0.0) || !x || !og || !out) return -1;
    const long rows = (long)B * H * L;
    for (long r = 0; r < rows; ++r) {
        const int h = (int)((r / L) % H);
        const double *xr = x + (size_t)r * dv;
        const float *gr = og + (size_t)r * dv;
        double *orow = out + (size_t)r * dv;
        double mean = 0.0;
        for (int i = 0; i < dv; ++i) mean += xr[i];
        mean /= dv;
        double var = 0.0;
        for (int i = 0; i < dv; ++i) var += (xr[i] - mean) * (xr[i] - mean);
        var /= dv;
        const double rstd = 1.0 / sqrt(var + eps);
        for (int i = 0; i < dv; ++i) {
            double y = (xr[i] - mean) * rstd;
            if (weight) y *= (double)weight[(size_t)h * dv + i];
            if (bias) y += (double)bias[(size_t)h * dv + i];
            orow[i] = or_swish((double)gr[i]) * y;
        }
    }
    return 0;
}

/*
 * oracle_backward: gradients of the forward pass (from S_0 = 0) with respect to
 * q, k, v and the per-channel gate g, given the gradient dout of its output.
 * The pages give no gradient; this is the chain rule applied to the recurrence
 * above, in fp64, one (b, h) at a time:
 *
 *   forward sweep   S_t, z_t as in or_sequence; num_t = qf^T S_t, den_t = qf.z_t
 *                   w_t = dout_t (unnormalised), or, with the normaliser,
 *                   w_t = dout_t / den_t and e_t = -(dout_t . out_t) / den_t
 *                   (out = num / den: d num = dout / den, d den = -dout.out/den)
 *                   dQ_t = S_t w_t + z_t e_t              (gradient of qf_t)
 *   reverse sweep   dS_t = diag(a_{t+1}) dS_{t+1} + qf_t w_t^T   (a_L taken as 0)
 *                   dz_t = a_{t+1} * dz_{t+1} + qf_t e_t
 *                   dK_t = dS_t v_t + dz_t                (gradient of kf_t)
 *                   dv_t = dS_t^T kf_t
 *   feature map     dq = dQ * phi'(q), dk = dK * phi'(k); elu+1: phi'(x) = 1
 *                   for x > 0, e^x otherwise
 *   channel gate    with B_t = sum_{r<=t} log a_r, every term of the output
 *                   carries e^{B_t - B_s} (query t, key s), so
 *                   dl/dB_t = qf_t * dQ_t - kf_t * dK_t, and log a_r enters
 *                   every B_t with t >= r: dl/dlog a_r = sum_{t>=r} dl/dB_t.
 *                   log a = logsigmoid(g) / 16 gives
 *                   dg_r = (dl/dlog a_r) * sigmoid(-g_r) / 16.
 *
 *   q, k, g, dq, dk, dg: [B,H,L,dk]; v, dout, dv: [B,H,L,dv]; gate as in
 *   oracle_forward; dg may be NULL (and is not written without the channel
 *   gate). Outputs are doubles. Returns 0, or -1 on a bad argument.
 */
int oracle_backward(const float *q, const float *k, const float *v,
                    const float *gate, const float *dout, int B, int H, int L,
                    int dk, int dv, int mode, double *dq, double *dkk,
                    double *dvv, double *dg, int nthreads)
{
    if (B < 0 || H < 0 || L < 0 || dk <= 0 || dv <= 0) return -1;
    if ((mode & (OR_GATE_HEAD | OR_GATE_CHANNEL)) && !gate) return -1;
    const int elu1 = (mode & OR_PHI_ELU1) != 0;
    const int norm = (mode & OR_NORMALIZE) != 0;
    const long nbh = (long)B * H;
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
    for (long bh = 0; bh < nbh; ++bh) {
        const size_t ok = (size_t)bh * L * dk, ov = (size_t)bh * L * dv;
        const float *qb = q + ok, *kb = k + ok, *vb = v + ov, *db = dout + ov;
        const float *gb = (mode & OR_GATE_CHANNEL) ? gate + ok : NULL;
        const double gamma = (mode & OR_GATE_HEAD) ? (double)gate[bh % H] : 1.0;
        /* per token: qf, kf, a (dk each), w (dv), e (1); the states */
        double *qf = (double *)malloc(sizeof(double) * ((size_t)L * (3 * (size_t)dk + dv + 1) +
                                                        2 * ((size_t)dk * dv + dk)));
        double *kf = qf + (size_t)L * dk, *a = kf + (size_t)L * dk, *w = a + (size_t)L * dk;
        double *e = w + (size_t)L * dv, *S = e + L, *z = S + (size_t)dk * dv;
        double *dS = z + dk, *dz = dS + (size_t)dk * dv;
        double *dQ = dq + ok, *dK = dkk + ok, *dV = dvv + ov;
        for (int t = 0; t < L; ++t)
            for (int i = 0; i < dk; ++i) {
                const size_t x = (size_t)t * dk + i;
                qf[x] = or_phi((double)qb[x], elu1);
                kf[x] = or_phi((double)kb[x], elu1);
                a[x] = gb ? exp(or_log_sigmoid((double)gb[x]) / 16.0) : gamma;
            }
        /* forward sweep */
        memset(S, 0, sizeof(double) * ((size_t)dk * dv + dk));
        for (int t = 0; t < L; ++t) {
            const double *qt = qf + (size_t)t * dk, *kt = kf + (size_t)t * dk, *at = a + (size_t)t * dk;
            for (int i = 0; i < dk; ++i) {
                for (int j = 0; j < dv; ++j)
                    S[(size_t)i * dv + j] = at[i] * S[(size_t)i * dv + j] + kt[i] * (double)vb[(size_t)t * dv + j];
                z[i] = at[i] * z[i] + kt[i];
            }
            double *wt = w + (size_t)t * dv;
            const float *dt = db + (size_t)t * dv;
            if (norm) {
                double den = 0.0, dot = 0.0;
                for (int i = 0; i < dk; ++i) den += qt[i] * z[i];
                for (int j = 0; j < dv; ++j) {
                    double num = 0.0;
                    for (int i = 0; i < dk; ++i) num += qt[i] * S[(size_t)i * dv + j];
                    dot += (double)dt[j] * (num / den);
                    wt[j] = (double)dt[j] / den;
                }
                e[t] = -dot / den;
            } else {
                for (int j = 0; j < dv; ++j) wt[j] = (double)dt[j];
                e[t] = 0.0;
            }
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) acc += S[(size_t)i * dv + j] * wt[j];
                dQ[(size_t)t * dk + i] = acc + z[i] * e[t];
            }
        }
        /* reverse sweep */
        memset(dS, 0, sizeof(double) * ((size_t)dk * dv + dk));
        for (int t = L - 1; t >= 0; --t) {
            const double *qt = qf + (size_t)t * dk, *kt = kf + (size_t)t * dk;
            const double *an = t + 1 < L ? a + (size_t)(t + 1) * dk : NULL;
            const double *wt = w + (size_t)t * dv;
            for (int i = 0; i < dk; ++i) {
                const double ai = an ? an[i] : 0.0;
                for (int j = 0; j < dv; ++j)
                    dS[(size_t)i * dv + j] = ai * dS[(size_t)i * dv + j] + qt[i] * wt[j];
                dz[i] = ai * dz[i] + qt[i] * e[t];
            }
            for (int i = 0; i < dk; ++i) {
                double acc = 0.0;
                for (int j = 0; j < dv; ++j) acc += dS[(size_t)i * dv + j] * (double)vb[(size_t)t * dv + j];
                dK[(size_t)t * dk + i] = acc + (norm ? dz[i] : 0.0);
            }
            for (int j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int i = 0; i < dk; ++i) acc += dS[(size_t)i * dv + j] * kt[i];
                dV[(size_t)t * dv + j] = acc;
            }
        }
        /* channel gate: reverse running sum of qf dQ - kf dK */
        if (gb && dg) {
            for (int i = 0; i < dk; ++i) {
                double c = 0.0;
                for (int t = L - 1; t >= 0; --t) {
                    const size_t x = (size_t)t * dk + i;
                    c += qf[x] * dQ[x] - kf[x] * dK[x];
                    const double gx = (double)gb[x];
                    /* sigmoid(-g), split so that neither branch overflows */
                    const double sm = gx >= 0.0 ? exp(-gx) / (1.0 + exp(-gx)) : 1.0 / (1.0 + exp(gx));
                    dg[ok + x] = c * sm / 16.0;
                }
            }
        }
        /* through the feature map */
        for (size_t x = 0; x < (size_t)L * dk; ++x) {
            if (elu1 && (double)qb[x] <= 0.0) dQ[x] *= exp((double)qb[x]);
            if (elu1 && (double)kb[x] <= 0.0) dK[x] *= exp((double)kb[x]);
        }
        free(qf);
    }
    (void)nthreads;
    return 0;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
