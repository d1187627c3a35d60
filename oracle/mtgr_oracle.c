/*
 * mtgr_oracle.c -- plain, slow, fp64 CPU oracle of one MTGR HSTU layer.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or helper with the CUDA path, and the CUDA path never calls it.
 *
 * Every function is the plain definition written out as loops, in fp64, with
 * no blocking, fusion or reordering beyond what the definition states.
 * OpenMP runs independent users (or independent rows) in parallel; each
 * output element is still summed in index order by one thread.
 *
 * Sources (web pages on MTGR, Meituan's generative-style ranking model):
 *  [P2] marovi.ai summary of arXiv 2505.18654, "Métodos": the block update
 *       Ṽ = silu(KᵀQ) / (N_U+N_S+N_R+N_I) · M · V, then GroupLN / MLP / residual.
 *  [P3] paper-daily.com "MTGR：美团外卖生成式推荐Scaling Law落地实践",
 *       "模型怎么搭": one linear + SiLU gives U, Q, K, V; attention weights
 *       SiLU(QKᵀ) without softmax; aggregate, normalise, gate with U, then a
 *       linear layer.
 *  [P4] fun-rec chapter 7.3, §7.3.3 (GLN formula) and §7.3.4 (three mask rules).
 *  [P1] zzxanthony.github.io MTGR post, §8 (GLN) and §9 (dynamic masking).
 *
 * Readings taken where the pages are open (each also listed in the design
 * notes): scores are scaled by 1/sqrt(d_h); n_u is the full segment length of
 * the user; GLN uses per-token statistics over d_model with per-group γ/β;
 * the gate is LayerNorm(O) ⊙ U with a plain (no affine) LayerNorm over all
 * H·d_h features; the block ends with x' = x + Y·W_o; there are no biases;
 * RealTime rows see RealTime keys with ts_j <= ts_i, candidate rows see
 * RealTime keys with ts_j < ts_i.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define G_USER 0
#define G_SEQ 1
#define G_RT 2
#define G_CAND 3

/* ------------------------------------------------------------------------ */
/* Dynamic mixed mask ([P4] §7.3.4 rules 1-3, [P1] §9): may query row i see   */
/* key j?  Both tokens belong to the same user segment.                      */
/* ------------------------------------------------------------------------ */
int orc_visible(int64_t i, int64_t j, const uint8_t* gid, const int64_t* ts) {
    const int gi = gid[i], gj = gid[j];
    if (gj == G_USER || gj == G_SEQ)       /* rule 1: static sequence, seen by all */
        return 1;
    if (gj == G_RT) {                      /* rule 2: realtime, causal in time */
        if (gi == G_RT) return ts[j] <= ts[i];
        if (gi == G_CAND) return ts[j] < ts[i];
        return 0;                          /* User/Seq rows precede the window */
    }
    return i == j;                         /* rule 3: a candidate sees only itself */
}

/* Per-row visible key counts and their total (integer metadata). */
void orc_visible_counts(int B, const int32_t* offsets, const uint8_t* gid, const int64_t* ts,
                        int32_t* cnt, int64_t* total) {
    int64_t tot = 0;
    for (int b = 0; b < B; ++b) {
        for (int64_t i = offsets[b]; i < offsets[b + 1]; ++i) {
            int32_t c = 0;
            for (int64_t j = offsets[b]; j < offsets[b + 1]; ++j) c += orc_visible(i, j, gid, ts);
            cnt[i] = c;
            tot += c;
        }
    }
    *total = tot;
}

static double silu(double s) { return s / (1.0 + exp(-s)); }
static double sigmoid(double s) { return 1.0 / (1.0 + exp(-s)); }

/* ------------------------------------------------------------------------ */
/* Attention core ([P2] block formula, [P3] "模型怎么搭"), per head h:         */
/*   s_ij = q_i·k_j / sqrt(d_h);  A_ij = M_ij · silu(s_ij) / n_u;             */
/*   O_i  = Σ_j A_ij v_j.                                                     */
/* q/k/v rows have stride ld (elements); head h occupies columns h*dh..+dh.  */
/* O is [T, H*dh] dense.  n_override > 0 replaces n_u (test-only, so that     */
/* invariants can be checked with the normaliser held fixed).               */
/* ------------------------------------------------------------------------ */
void orc_attn_core_fwd(int B, const int32_t* offsets, const uint8_t* gid, const int64_t* ts,
                       int H, int dh, const double* q, const double* k, const double* v,
                       int64_t ld, double n_override, double* O) {
    const int HD = H * dh;
    const double c = 1.0 / sqrt((double)dh);
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const int64_t s0 = offsets[b], s1 = offsets[b + 1];
        const double nu = n_override > 0 ? n_override : (double)(s1 - s0);
        double* acc = (double*)malloc(sizeof(double) * dh);
        for (int64_t i = s0; i < s1; ++i) {
            for (int h = 0; h < H; ++h) {
                for (int d = 0; d < dh; ++d) acc[d] = 0.0;
                const double* qi = q + i * ld + h * dh;
                for (int64_t j = s0; j < s1; ++j) {
                    if (!orc_visible(i, j, gid, ts)) continue;
                    const double* kj = k + j * ld + h * dh;
                    const double* vj = v + j * ld + h * dh;
                    double s = 0.0;
                    for (int d = 0; d < dh; ++d) s += qi[d] * kj[d];
                    s *= c;
                    const double a = silu(s) / nu;
                    for (int d = 0; d < dh; ++d) acc[d] += a * vj[d];
                }
                for (int d = 0; d < dh; ++d) O[i * HD + h * dh + d] = acc[d];
            }
        }
        free(acc);
    }
}

/* Backward of the attention core for upstream dO [T, H*dh]:                  */
/*   dv_j += A_ij dO_i;  dA_ij = dO_i·v_j;  ds_ij = dA_ij silu'(s_ij) / n_u;   */
/*   dq_i += ds_ij k_j / sqrt(d_h);  dk_j += ds_ij q_i / sqrt(d_h),            */
/* with silu'(s) = σ(s)(1 + s(1-σ(s))).  Outputs use row stride ldg and are   */
/* overwritten for every row of every segment.                               */
void orc_attn_core_bwd(int B, const int32_t* offsets, const uint8_t* gid, const int64_t* ts,
                       int H, int dh, const double* q, const double* k, const double* v,
                       int64_t ld, double n_override, const double* dO,
                       double* dq, double* dk, double* dv, int64_t ldg) {
    const int HD = H * dh;
    const double c = 1.0 / sqrt((double)dh);
#pragma omp parallel for schedule(dynamic, 1)
    for (int b = 0; b < B; ++b) {
        const int64_t s0 = offsets[b], s1 = offsets[b + 1];
        const double nu = n_override > 0 ? n_override : (double)(s1 - s0);
        for (int64_t i = s0; i < s1; ++i)
            for (int h = 0; h < H; ++h)
                for (int d = 0; d < dh; ++d) {
                    dq[i * ldg + h * dh + d] = 0.0;
                    dk[i * ldg + h * dh + d] = 0.0;
                    dv[i * ldg + h * dh + d] = 0.0;
                }
        for (int64_t i = s0; i < s1; ++i) {
            for (int h = 0; h < H; ++h) {
                const double* qi = q + i * ld + h * dh;
                const double* gi = dO + i * HD + h * dh;
                for (int64_t j = s0; j < s1; ++j) {
                    if (!orc_visible(i, j, gid, ts)) continue;
                    const double* kj = k + j * ld + h * dh;
                    const double* vj = v + j * ld + h * dh;
                    double s = 0.0, dA = 0.0;
                    for (int d = 0; d < dh; ++d) s += qi[d] * kj[d];
                    s *= c;
                    for (int d = 0; d < dh; ++d) dA += gi[d] * vj[d];
                    const double sg = sigmoid(s);
                    const double a = s * sg / nu;
                    const double ds = dA * sg * (1.0 + s * (1.0 - sg)) / nu;
                    for (int d = 0; d < dh; ++d) {
                        dv[j * ldg + h * dh + d] += a * gi[d];
                        dq[i * ldg + h * dh + d] += ds * c * kj[d];
                        dk[j * ldg + h * dh + d] += ds * c * qi[d];
                    }
                }
            }
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Gate ([P3] "模型怎么搭": normalise the aggregate, multiply by U):           */
/*   Y_t = LN(O_t) ⊙ U_t, LN over the n features of row t, no affine,        */
/*   biased variance, eps inside the square root.                            */
/* ------------------------------------------------------------------------ */
void orc_ln_gate_fwd(int64_t T, int n, const double* O, const double* U, int64_t ldu, double eps,
                     double* Y, double* mean, double* rstd) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* o = O + t * n;
        double mu = 0.0, var = 0.0;
        for (int f = 0; f < n; ++f) mu += o[f];
        mu /= n;
        for (int f = 0; f < n; ++f) var += (o[f] - mu) * (o[f] - mu);
        var /= n;
        const double r = 1.0 / sqrt(var + eps);
        for (int f = 0; f < n; ++f) Y[t * n + f] = (o[f] - mu) * r * U[t * ldu + f];
        if (mean) mean[t] = mu;
        if (rstd) rstd[t] = r;
    }
}

/* Backward of the gate: with ô = (O-μ)r, dU = dY ⊙ ô, dô = dY ⊙ U,
 * dO = r (dô - mean(dô) - ô mean(dô ⊙ ô)).  dU uses row stride ldg. */
void orc_ln_gate_bwd(int64_t T, int n, const double* dY, const double* O, const double* U, int64_t ldu,
                     double eps, double* dO, double* dU, int64_t ldg) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* o = O + t * n;
        double mu = 0.0, var = 0.0;
        for (int f = 0; f < n; ++f) mu += o[f];
        mu /= n;
        for (int f = 0; f < n; ++f) var += (o[f] - mu) * (o[f] - mu);
        var /= n;
        const double r = 1.0 / sqrt(var + eps);
        double m1 = 0.0, m2 = 0.0;
        for (int f = 0; f < n; ++f) {
            const double oh = (o[f] - mu) * r;
            const double g = dY[t * n + f] * U[t * ldu + f];
            m1 += g;
            m2 += g * oh;
        }
        m1 /= n;
        m2 /= n;
        for (int f = 0; f < n; ++f) {
            const double oh = (o[f] - mu) * r;
            const double g = dY[t * n + f] * U[t * ldu + f];
            dU[t * ldg + f] = dY[t * n + f] * oh;
            dO[t * n + f] = r * (g - m1 - oh * m2);
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Group LayerNorm ([P4] §7.3.3: GLN(x_i) = (x_i-μ)/σ · γ_g(i) + β_g(i);      */
/* [P3] "模型怎么搭": each token class gets its own normalisation parameters). */
/* Statistics are per token over its D features; γ, β are [4, D].           */
/* ------------------------------------------------------------------------ */
void orc_gln_fwd(int64_t T, int D, const double* x, const uint8_t* gid, const double* gamma,
                 const double* beta, double eps, double* y, double* mean, double* rstd) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* xr = x + t * D;
        const int g = gid[t];
        double mu = 0.0, var = 0.0;
        for (int f = 0; f < D; ++f) mu += xr[f];
        mu /= D;
        for (int f = 0; f < D; ++f) var += (xr[f] - mu) * (xr[f] - mu);
        var /= D;
        const double r = 1.0 / sqrt(var + eps);
        for (int f = 0; f < D; ++f) y[t * D + f] = (xr[f] - mu) * r * gamma[g * D + f] + beta[g * D + f];
        if (mean) mean[t] = mu;
        if (rstd) rstd[t] = r;
    }
}

/* GLN backward: x̂ = (x-μ)r, dx̂ = dy ⊙ γ_g, dx = r (dx̂ - mean(dx̂) - x̂ mean(dx̂ ⊙ x̂)),
 * dγ_g = Σ_{t in g} dy_t ⊙ x̂_t, dβ_g = Σ_{t in g} dy_t (summed in token order). */
void orc_gln_bwd(int64_t T, int D, const double* dy, const double* x, const uint8_t* gid,
                 const double* gamma, double eps, double* dx, double* dgamma, double* dbeta) {
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < T; ++t) {
        const double* xr = x + t * D;
        const int g = gid[t];
        double mu = 0.0, var = 0.0;
        for (int f = 0; f < D; ++f) mu += xr[f];
        mu /= D;
        for (int f = 0; f < D; ++f) var += (xr[f] - mu) * (xr[f] - mu);
        var /= D;
        const double r = 1.0 / sqrt(var + eps);
        double m1 = 0.0, m2 = 0.0;
        for (int f = 0; f < D; ++f) {
            const double xh = (xr[f] - mu) * r;
            const double gx = dy[t * D + f] * gamma[g * D + f];
            m1 += gx;
            m2 += gx * xh;
        }
        m1 /= D;
        m2 /= D;
        for (int f = 0; f < D; ++f) {
            const double xh = (xr[f] - mu) * r;
            const double gx = dy[t * D + f] * gamma[g * D + f];
            dx[t * D + f] = r * (gx - m1 - xh * m2);
        }
    }
    /* Parameter gradients: each feature column summed over tokens in order. */
    double* mus = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
    double* rs = (double*)malloc(sizeof(double) * (T > 0 ? T : 1));
    for (int64_t t = 0; t < T; ++t) {
        const double* xr = x + t * D;
        double mu = 0.0, var = 0.0;
        for (int e = 0; e < D; ++e) mu += xr[e];
        mu /= D;
        for (int e = 0; e < D; ++e) var += (xr[e] - mu) * (xr[e] - mu);
        var /= D;
        mus[t] = mu;
        rs[t] = 1.0 / sqrt(var + eps);
    }
#pragma omp parallel for schedule(static)
    for (int f = 0; f < D; ++f) {
        double sg[4] = {0, 0, 0, 0}, sb[4] = {0, 0, 0, 0};
        for (int64_t t = 0; t < T; ++t) {
            const int g = gid[t];
            sg[g] += dy[t * D + f] * (x[t * D + f] - mus[t]) * rs[t];
            sb[g] += dy[t * D + f];
        }
        for (int g = 0; g < 4; ++g) {
            dgamma[g * D + f] = sg[g];
            dbeta[g * D + f] = sb[g];
        }
    }
    free(mus);
    free(rs);
}

/* ------------------------------------------------------------------------ */
/* Plain matrix products, summed over k in index order.                      */
/* ------------------------------------------------------------------------ */
/* C[M,N] = A[M,K] · B[K,N] */
void orc_matmul(int64_t M, int64_t N, int64_t K, const double* A, const double* Bm, double* C) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double* c = C + m * N;
        for (int64_t n = 0; n < N; ++n) c[n] = 0.0;
        for (int64_t kk = 0; kk < K; ++kk) {
            const double a = A[m * K + kk];
            const double* b = Bm + kk * N;
            for (int64_t n = 0; n < N; ++n) c[n] += a * b[n];
        }
    }
}

/* C[M,N] = A[M,K] · B[N,K]ᵀ */
void orc_matmul_nt(int64_t M, int64_t N, int64_t K, const double* A, const double* Bm, double* C) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m)
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t kk = 0; kk < K; ++kk) s += A[m * K + kk] * Bm[n * K + kk];
            C[m * N + n] = s;
        }
}

/* C[M,N] = A[K,M]ᵀ · B[K,N] */
void orc_matmul_tn(int64_t M, int64_t N, int64_t K, const double* A, const double* Bm, double* C) {
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        double* c = C + m * N;
        for (int64_t n = 0; n < N; ++n) c[n] = 0.0;
        for (int64_t kk = 0; kk < K; ++kk) {
            const double a = A[kk * M + m];
            const double* b = Bm + kk * N;
            for (int64_t n = 0; n < N; ++n) c[n] += a * b[n];
        }
    }
}

/* ------------------------------------------------------------------------ */
/* One HSTU layer ([P3] "模型怎么搭", [P5] "统一 HSTU 编码 + Group LayerNorm"):   */
/*   xn = GLN(x);  z = xn · W_uqkv;  [U|Q|K|V] = silu(z);                     */
/*   O = attention core;  Y = LN(O) ⊙ U;  x' = x + Y · W_o.                  */
/* W_uqkv is [D, 4HD] with column blocks U, Q, K, V (each head-major);       */
/* W_o is [HD, D].  Saved intermediates are written when the pointer is set. */
/* ------------------------------------------------------------------------ */
void orc_layer_fwd(int B, const int32_t* offsets, const uint8_t* gid, const int64_t* ts,
                   int64_t T, int D, int H, int dh, const double* x, const double* w_uqkv,
                   const double* w_o, const double* gamma, const double* beta, double eps_gln,
                   double eps_ln, double* x_out, double* xn_s, double* z_s, double* o_s, double* y_s) {
    const int HD = H * dh;
    double* xn = (double*)malloc(sizeof(double) * T * D);
    double* z = (double*)malloc(sizeof(double) * T * 4 * HD);
    double* a = (double*)malloc(sizeof(double) * T * 4 * HD);
    double* O = (double*)malloc(sizeof(double) * T * HD);
    double* Y = (double*)malloc(sizeof(double) * T * HD);
    orc_gln_fwd(T, D, x, gid, gamma, beta, eps_gln, xn, 0, 0);
    orc_matmul(T, 4 * HD, D, xn, w_uqkv, z);
    for (int64_t e = 0; e < T * 4 * HD; ++e) a[e] = silu(z[e]);
    /* U = a[:, 0:HD], Q = a[:, HD:2HD], K = a[:, 2HD:3HD], V = a[:, 3HD:4HD] */
    orc_attn_core_fwd(B, offsets, gid, ts, H, dh, a + HD, a + 2 * HD, a + 3 * HD, 4 * HD, 0.0, O);
    orc_ln_gate_fwd(T, HD, O, a, 4 * HD, eps_ln, Y, 0, 0);
    orc_matmul(T, D, HD, Y, w_o, x_out);
    for (int64_t e = 0; e < T * D; ++e) x_out[e] += x[e];
    if (xn_s) memcpy(xn_s, xn, sizeof(double) * T * D);
    if (z_s) memcpy(z_s, z, sizeof(double) * T * 4 * HD);
    if (o_s) memcpy(o_s, O, sizeof(double) * T * HD);
    if (y_s) memcpy(y_s, Y, sizeof(double) * T * HD);
    free(xn); free(z); free(a); free(O); free(Y);
}

/* Backward of one layer for upstream dx_out:
 *   dY = dx'·W_oᵀ, dW_o = Yᵀ·dx';  (dO, dU) = gate bwd;  (dQ, dK, dV) = core bwd;
 *   dz = [dU|dQ|dK|dV] ⊙ silu'(z);  dW_uqkv = xnᵀ·dz;  dxn = dz·W_uqkvᵀ;
 *   (dx_gln, dγ, dβ) = GLN bwd(dxn);  dx = dx' + dx_gln. */
void orc_layer_bwd(int B, const int32_t* offsets, const uint8_t* gid, const int64_t* ts,
                   int64_t T, int D, int H, int dh, const double* x, const double* w_uqkv,
                   const double* w_o, const double* gamma, const double* beta, double eps_gln,
                   double eps_ln, const double* dx_out, double* dx, double* dw_uqkv, double* dw_o,
                   double* dgamma, double* dbeta) {
    const int HD = H * dh;
    const int64_t N4 = 4 * (int64_t)HD;
    double* xn = (double*)malloc(sizeof(double) * T * D);
    double* z = (double*)malloc(sizeof(double) * T * N4);
    double* a = (double*)malloc(sizeof(double) * T * N4);
    double* O = (double*)malloc(sizeof(double) * T * HD);
    double* Y = (double*)malloc(sizeof(double) * T * HD);
    double* xo = (double*)malloc(sizeof(double) * T * D);
    double* dY = (double*)malloc(sizeof(double) * T * HD);
    double* dO = (double*)malloc(sizeof(double) * T * HD);
    double* da = (double*)malloc(sizeof(double) * T * N4);
    double* dxn = (double*)malloc(sizeof(double) * T * D);
    orc_layer_fwd(B, offsets, gid, ts, T, D, H, dh, x, w_uqkv, w_o, gamma, beta, eps_gln, eps_ln,
                  xo, xn, z, O, Y);
    for (int64_t e = 0; e < T * N4; ++e) a[e] = silu(z[e]);
    orc_matmul_nt(T, HD, D, dx_out, w_o, dY);
    orc_matmul_tn(HD, D, T, Y, dx_out, dw_o);
    orc_ln_gate_bwd(T, HD, dY, O, a, N4, eps_ln, dO, da, N4);
    orc_attn_core_bwd(B, offsets, gid, ts, H, dh, a + HD, a + 2 * HD, a + 3 * HD, N4, 0.0, dO,
                      da + HD, da + 2 * HD, da + 3 * HD, N4);
    for (int64_t e = 0; e < T * N4; ++e) {
        const double sg = sigmoid(z[e]);
        da[e] *= sg * (1.0 + z[e] * (1.0 - sg));
    }
    orc_matmul_tn(D, N4, T, xn, da, dw_uqkv);
    orc_matmul_nt(T, D, N4, da, w_uqkv, dxn);
    orc_gln_bwd(T, D, dxn, x, gid, gamma, eps_gln, dx, dgamma, dbeta);
    for (int64_t e = 0; e < T * D; ++e) dx[e] += dx_out[e];
    (void)beta;
    free(xn); free(z); free(a); free(O); free(Y); free(xo); free(dY); free(dO); free(da); free(dxn);
}
