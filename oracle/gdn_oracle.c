/*
 * gdn_oracle.c -- fp64 CPU oracle for the Gated DeltaNet linear-attention layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, literal definition the GPU
 * library is checked against.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg load it.  It shares no code, header or constant with
 * the CUDA path, and the CUDA path never calls it.
 *
 * What it follows: the MNN discussion "MNN Model Support: Qwen3.5", section 1.2
 * (Algorithm Principles: the five steps over qkv [B, D, L], gate and beta
 * [B, L, H], conv_weight [D, 1, K]), section 1.3 (Reverse GQA by
 * repeat_interleave) and section 1.4 (the conv state [B, D, K-1] and the
 * recurrent state [B, H, d_k, d_v], zeroed at the start and carried across
 * steps).
 *
 * Readings where the page leaves a step open:
 *   - the conv is a cross-correlation in PyTorch conv1d orientation on [D,1,K]
 *     weights: w[d][K-1] multiplies the newest sample; no bias;
 *   - the conv state holds the raw (pre-conv) inputs of the last K-1 steps,
 *     oldest first;
 *   - SiLU applies to all D channels;
 *   - channels split as Q = [0, Hk*dk), K = [Hk*dk, 2*Hk*dk), V = the rest,
 *     head-major inside each range;
 *   - value head h reads key head h / (Hv/Hk) (repeat_interleave, not tiling);
 *   - L2 normalisation is x * 1/sqrt(sum x^2 + eps);
 *   - the output of token t reads the state after token t's update.
 *
 * Everything is double precision, single-threaded, with no blocking or
 * reordering: each loop is the formula it implements.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <string.h>

/* ---- Step 1: depthwise causal Conv1D + SiLU (section 1.2, Step 1) -------- */
/*
 * One sequence.  Let xt = [state_in[d][0..K-2], x[d][0..L-1]] (length K-1+L).
 * y[d][t] = silu( sum_{j=0}^{K-1} w[d][j] * xt[t+j] ),  silu(a) = a / (1 + e^-a).
 * state_out[d] = the last K-1 entries of xt.
 * x, y: [D][L]; w: [D][K]; state_in, state_out: [D][K-1] (they may alias).
 * conv_snap (optional): [L][D][K-1], the window after each token t,
 * i.e. xt[t+1 .. t+K-1].
 */
void gdn_oracle_conv1d_silu(int64_t D, int64_t K, int64_t L,
                            const double *x, const double *w,
                            const double *state_in, double *y,
                            double *state_out, double *conv_snap)
{
    const int64_t P = K - 1 + L;          /* length of xt */
    for (int64_t d = 0; d < D; ++d) {
        for (int64_t t = 0; t < L; ++t) {
            double acc = 0.0;
            for (int64_t j = 0; j < K; ++j) {
                int64_t p = t + j;                 /* index into xt */
                double xv = (p < K - 1) ? state_in[d * (K - 1) + p]
                                        : x[d * L + (p - (K - 1))];
                acc += w[d * K + j] * xv;
            }
            y[d * L + t] = acc / (1.0 + exp(-acc));
        }
        if (conv_snap) {
            for (int64_t t = 0; t < L; ++t)
                for (int64_t i = 0; i < K - 1; ++i) {
                    int64_t p = t + 1 + i;
                    conv_snap[(t * D + d) * (K - 1) + i] =
                        (p < K - 1) ? state_in[d * (K - 1) + p]
                                    : x[d * L + (p - (K - 1))];
                }
        }
        for (int64_t i = 0; i < K - 1; ++i) {
            int64_t p = P - (K - 1) + i;
            state_out[d * (K - 1) + i] = (p < K - 1) ? state_in[d * (K - 1) + p]
                                                     : x[d * L + (p - (K - 1))];
        }
    }
}

/* ---- Steps 2-4: split, reverse GQA, L2 norm, scale (section 1.2 Steps 2-4,
 *      section 1.3) ---------------------------------------------------------- */
/*
 * y: [D][L] conv output of one sequence.  Writes, per token t and value head h:
 *   q[t][h][i] = Q channel (h/f)*dk + i, k[t][h][i] = K channel (h/f)*dk + i,
 *   v[t][h][j] = V channel h*dv + j, with f = Hv/Hk;
 * then, when use_l2 is set, q and k are divided by sqrt(sum of squares + eps)
 * over the dk entries of their head; finally q is divided by sqrt(dk).
 * q, k: [L][Hv][dk]; v: [L][Hv][dv].
 */
void gdn_oracle_split_norm_scale(int64_t Hk, int64_t Hv, int64_t dk, int64_t dv,
                                 int64_t L, int use_l2, double eps,
                                 const double *y, double *q, double *k, double *v)
{
    const int64_t f = Hv / Hk;
    const int64_t q0 = 0, k0 = Hk * dk, v0 = 2 * Hk * dk;
    for (int64_t t = 0; t < L; ++t) {
        for (int64_t h = 0; h < Hv; ++h) {
            const int64_t hk = h / f;           /* repeat_interleave(f) */
            double *qt = q + (t * Hv + h) * dk;
            double *kt = k + (t * Hv + h) * dk;
            double *vt = v + (t * Hv + h) * dv;
            for (int64_t i = 0; i < dk; ++i) {
                qt[i] = y[(q0 + hk * dk + i) * L + t];
                kt[i] = y[(k0 + hk * dk + i) * L + t];
            }
            for (int64_t j = 0; j < dv; ++j)
                vt[j] = y[(v0 + h * dv + j) * L + t];
            if (use_l2) {
                double sq = 0.0, sk = 0.0;
                for (int64_t i = 0; i < dk; ++i) {
                    sq += qt[i] * qt[i];
                    sk += kt[i] * kt[i];
                }
                const double nq = sqrt(sq + eps), nk = sqrt(sk + eps);
                for (int64_t i = 0; i < dk; ++i) {
                    qt[i] = qt[i] / nq;
                    kt[i] = kt[i] / nk;
                }
            }
            const double s = sqrt((double)dk);
            for (int64_t i = 0; i < dk; ++i)
                qt[i] = qt[i] / s;
        }
    }
}

/* ---- Step 5: gated delta rule (section 1.2, Step 5) ----------------------- */
/*
 * For each value head h, starting from S = S_in[h] ([dk][dv], row i = key dim),
 * and for t = 0..L-1, in the page's order:
 *   S      = S * exp(g[t][h])
 *   vpred  = S^T k_t                      (vpred[j] = sum_i S[i][j] k_t[i])
 *   delta  = beta[t][h] * (v_t - vpred)
 *   S      = S + k_t delta^T              (S[i][j] += k_t[i] delta[j])
 *   o_t    = S^T q_t                      (o[t][h][j] = sum_i S[i][j] q_t[i])
 * S_out[h] = S after the last token; S_snap[t][h] (optional) = S after token t.
 * q, k: [L][H][dk]; v: [L][H][dv]; g, beta: [L][H]; S_in, S_out: [H][dk][dv];
 * o: [L][H][dv]; S_snap: [L][H][dk][dv].  S_in and S_out may alias.
 */
void gdn_oracle_delta_rule(int64_t H, int64_t dk, int64_t dv, int64_t L,
                           const double *q, const double *k, const double *v,
                           const double *g, const double *beta,
                           const double *S_in, double *o, double *S_out,
                           double *S_snap, double *work /* [dk*dv + dv + dv] */)
{
    double *S = work;
    double *vpred = work + dk * dv;
    double *delta = vpred + dv;
    for (int64_t h = 0; h < H; ++h) {
        memcpy(S, S_in + h * dk * dv, sizeof(double) * (size_t)(dk * dv));
        for (int64_t t = 0; t < L; ++t) {
            const double *kt = k + (t * H + h) * dk;
            const double *qt = q + (t * H + h) * dk;
            const double *vt = v + (t * H + h) * dv;
            const double decay = exp(g[t * H + h]);
            const double b = beta[t * H + h];
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j)
                    S[i * dv + j] = S[i * dv + j] * decay;
            for (int64_t j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < dk; ++i)
                    acc += S[i * dv + j] * kt[i];
                vpred[j] = acc;
            }
            for (int64_t j = 0; j < dv; ++j)
                delta[j] = b * (vt[j] - vpred[j]);
            for (int64_t i = 0; i < dk; ++i)
                for (int64_t j = 0; j < dv; ++j)
                    S[i * dv + j] = S[i * dv + j] + kt[i] * delta[j];
            for (int64_t j = 0; j < dv; ++j) {
                double acc = 0.0;
                for (int64_t i = 0; i < dk; ++i)
                    acc += S[i * dv + j] * qt[i];
                o[(t * H + h) * dv + j] = acc;
            }
            if (S_snap)
                memcpy(S_snap + (t * H + h) * dk * dv, S,
                       sizeof(double) * (size_t)(dk * dv));
        }
        memcpy(S_out + h * dk * dv, S, sizeof(double) * (size_t)(dk * dv));
    }
}

/* ---- All five steps for one sequence -------------------------------------- */
/*
 * x: [D][L] raw qkv of the sequence; w: [D][K]; conv_in/conv_out: [D][K-1];
 * S_in/S_out: [Hv][dk][dv]; g, beta: [L][Hv]; o: [L][Hv][dv];
 * conv_snap: [L][D][K-1] or NULL; S_snap: [L][Hv][dk][dv] or NULL.
 * work: caller scratch of at least D*L + L*Hv*(2*dk+dv) + dk*dv + 2*dv doubles.
 */
void gdn_oracle_forward(int64_t Hk, int64_t Hv, int64_t dk, int64_t dv, int64_t K,
                        int use_l2, double eps, int64_t L,
                        const double *x, const double *w, const double *conv_in,
                        const double *S_in, const double *g, const double *beta,
                        double *o, double *conv_out, double *S_out,
                        double *conv_snap, double *S_snap, double *work)
{
    const int64_t D = 2 * Hk * dk + Hv * dv;
    double *y = work;
    double *q = y + D * L;
    double *kk = q + L * Hv * dk;
    double *v = kk + L * Hv * dk;
    double *rw = v + L * Hv * dv;
    gdn_oracle_conv1d_silu(D, K, L, x, w, conv_in, y, conv_out, conv_snap);
    gdn_oracle_split_norm_scale(Hk, Hv, dk, dv, L, use_l2, eps, y, q, kk, v);
    gdn_oracle_delta_rule(Hv, dk, dv, L, q, kk, v, g, beta, S_in, o, S_out, S_snap, rw);
}

/* ---- Gate parameterisation (section 1.2, after Step 5) ------------------- */
/*
 * From the raw projections a, b [n][H] and the per-head parameters A_log,
 * dt_bias [H]:
 *   gate[t][h] = -exp(A_log[h]) * softplus(a[t][h] + dt_bias[h]),
 *   beta[t][h] = sigmoid(b[t][h]) = 1 / (1 + exp(-b[t][h])),
 * with softplus(x) = log(1 + exp(x)), written as max(x, 0) + log1p(exp(-|x|))
 * (the same number, without overflow for large x).
 */
void gdn_oracle_gate_beta(int64_t n, int64_t H, const double *a, const double *b,
                          const double *A_log, const double *dt_bias,
                          double *gate, double *beta) {
    for (int64_t t = 0; t < n; ++t)
        for (int64_t h = 0; h < H; ++h) {
            const double x = a[t * H + h] + dt_bias[h];
            const double sp = (x > 0.0 ? x : 0.0) + log1p(exp(-fabs(x)));
            gate[t * H + h] = -exp(A_log[h]) * sp;
            beta[t * H + h] = 1.0 / (1.0 + exp(-b[t * H + h]));
        }
}

/* ---- Gated RMSNorm of the layer output (section 2) ----------------------- */
/*
 * For each of `rows` rows of n values:
 *   y[r][j] = weight[j] * o[r][j] / sqrt(mean_i o[r][i]^2 + eps) * silu(z[r][j]),
 * silu(a) = a / (1 + e^-a).  The rows are the (token, value head) pairs of the
 * layer output; n = head_v_dim.
 */
void gdn_oracle_gated_rmsnorm(int64_t rows, int64_t n, const double *o, const double *z,
                              const double *weight, double eps, double *y) {
    for (int64_t r = 0; r < rows; ++r) {
        double sq = 0.0;
        for (int64_t j = 0; j < n; ++j) sq += o[r * n + j] * o[r * n + j];
        const double rms = sqrt(sq / (double)n + eps);
        for (int64_t j = 0; j < n; ++j) {
            const double zz = z[r * n + j];
            y[r * n + j] = weight[j] * (o[r * n + j] / rms) * (zz / (1.0 + exp(-zz)));
        }
    }
}

int64_t gdn_oracle_forward_work_doubles(int64_t Hk, int64_t Hv, int64_t dk,
                                        int64_t dv, int64_t L)
{
    const int64_t D = 2 * Hk * dk + Hv * dv;
    return D * L + L * Hv * (2 * dk + dv) + dk * dv + 2 * dv;
}
