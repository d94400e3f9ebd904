// GGD-BAM attention oracle: a plain, slow, fp64 CPU statement of what the GPU
// library computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
// the CPU-baseline leg of the benchmark call it; the library itself never does.
// It shares no code, header or constant with the CUDA path.
//
// Sources (page title, section / equation):
//  * "Bayesian Attention Mechanism" technical summary (gist.science, 2505.22842),
//    "Solution Proposee : GGD-BAM": the per-head Generalized-Gaussian bias
//    b = -|(offset - mu) / alpha|^beta, and the SSMax note ("dynamic logit
//    rescaling") in the same section.
//  * BAM repository README (ArthurSBianchessi/BAM), "Implementation Details":
//    the bias equation with eps = 1e-5 and the AttentionPrior module.
//  * "ALiBi: Attention with Linear Biases" (creativeworksofknowledge), "Code":
//    scores = Q K^T / sqrt(d_k) + bias, softmax over keys, weights @ V.
//  * "NNX ALiBi-Style Attention" (crackedaicode), first section: the scaled
//    score dot(Q,K)/sqrt(Dh) minus the distance penalty, non-causal.
//
// Readings taken where the pages are silent or disagree (each is also listed
// in the design notes):
//  * offset: d = i - j (query minus key) and u = |d - mu|; mu > 0 moves the
//    peak of the prior into the visible past.
//  * eps: for beta <= 0, u is clamped to max(u, eps); for beta > 0 no eps.
//    0^beta = 0 for beta > 0.
//  * SSMax: z_ij = s_h * ln(n_i) * q_i.k_j / sqrt(D) + b_ij with n_i the
//    number of visible keys (i+1 causal, T non-causal, Tkv for decode); the
//    bias is not rescaled.  Without SSMax z_ij = q_i.k_j / sqrt(D) + b_ij.
//  * backward: the pages give none; the plain chain rule of L = sum(O * dO).
//    At u = 0 (beta > 0) the contributions to dalpha, dbeta, dmu are 0 (their
//    limits, with sgn(0) = 0); where the eps clamp is active du/dmu = 0.
//  * theta prior (prior = 1): the repository README's own parameterisation,
//    "Implementation Details" (the bias equation and AttentionPrior.forward):
//    b = -exp(theta_alpha) * (|d - mu| + eps)^theta_beta with
//    mu = exp(theta_mu) - exp(-theta_mu) and eps added for every theta_beta;
//    the gradients are with respect to theta_alpha, theta_beta, theta_mu.
//    With eps = 0 and |d - mu| = 0 the value is 0 for theta_beta > 0.
//
// Layouts: q, k, v, o, dO, dq, dk, dv are [B, H, T, D] row-major doubles;
// lse is [B, H, T] (natural log); per-head parameters are double[H].
// The decode entry takes q [B, H, D] and a cache [B, H, Tkv, D].

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

namespace {

struct Params {
    const double* alpha;  // theta_alpha when prior == 1
    const double* beta;   // theta_beta when prior == 1
    const double* mu;     // theta_mu when prior == 1
    const double* s;      // SSMax scale, read only when ssmax != 0
    double eps;
    int causal;
    int ssmax;
    int prior;  // 0: -(u/alpha)^beta with the eps clamp; 1: theta prior
};

// |d - mu|, clamped to eps for beta <= 0.  Returns whether the clamp is active.
double offset_u(double d, double mu, double beta, double eps, bool* clamped) {
    double u = std::fabs(d - mu);
    bool c = false;
    if (beta <= 0.0 && u < eps) {
        u = eps;
        c = true;
    }
    if (clamped) *clamped = c;
    return u;
}

// GGD-BAM bias b(d) = -(u / alpha)^beta.
double bias(double d, double alpha, double beta, double mu, double eps) {
    double u = offset_u(d, mu, beta, eps, nullptr);
    if (u == 0.0) return 0.0;  // beta > 0 here: 0^beta = 0
    return -std::pow(u / alpha, beta);
}

// Partial derivatives of b with respect to alpha, beta and mu, by hand:
//   db/dalpha = beta * (u/alpha)^beta / alpha
//   db/dbeta  = -(u/alpha)^beta * ln(u/alpha)
//   db/du     = -beta * (u/alpha)^(beta-1) / alpha,  du/dmu = -sgn(d - mu)
void bias_grad(double d, double alpha, double beta, double mu, double eps,
               double* da, double* db, double* dm) {
    bool clamped = false;
    double u = offset_u(d, mu, beta, eps, &clamped);
    if (u == 0.0) {
        *da = 0.0;
        *db = 0.0;
        *dm = 0.0;
        return;
    }
    double r = u / alpha;
    double rb = std::pow(r, beta);
    *da = beta * rb / alpha;
    *db = -rb * std::log(r);
    if (clamped) {
        *dm = 0.0;
    } else {
        double dbdu = -beta * std::pow(r, beta - 1.0) / alpha;
        double sgn = (d - mu > 0.0) ? 1.0 : ((d - mu < 0.0) ? -1.0 : 0.0);
        *dm = dbdu * (-sgn);
    }
}

// theta prior: b = -exp(ta) * w^tb, w = |d - mu| + eps, mu = exp(tm) - exp(-tm).
double theta_mu_value(double tm) { return std::exp(tm) - std::exp(-tm); }

double bias_theta(double d, double ta, double tb, double tm, double eps) {
    double w = std::fabs(d - theta_mu_value(tm)) + eps;
    if (w == 0.0) return 0.0;  // eps == 0 at d == mu, tb > 0: 0^tb = 0
    return -std::exp(ta) * std::pow(w, tb);
}

// Its partial derivatives, by hand:
//   db/dta = b,   db/dtb = b * ln(w),
//   db/dw = tb * b / w,  dw/dmu = -sgn(d - mu),  dmu/dtm = exp(tm) + exp(-tm).
void bias_theta_grad(double d, double ta, double tb, double tm, double eps,
                     double* gta, double* gtb, double* gtm) {
    double mu = theta_mu_value(tm);
    double w = std::fabs(d - mu) + eps;
    if (w == 0.0) {
        *gta = 0.0;
        *gtb = 0.0;
        *gtm = 0.0;
        return;
    }
    double b = -std::exp(ta) * std::pow(w, tb);
    *gta = b;
    *gtb = b * std::log(w);
    double sgn = (d - mu > 0.0) ? 1.0 : ((d - mu < 0.0) ? -1.0 : 0.0);
    *gtm = (tb * b / w) * (-sgn) * (std::exp(tm) + std::exp(-tm));
}

// The bias and its three partials for head h under either prior.
double bias_of(const Params& p, int h, double d) {
    if (p.prior) return bias_theta(d, p.alpha[h], p.beta[h], p.mu[h], p.eps);
    return bias(d, p.alpha[h], p.beta[h], p.mu[h], p.eps);
}

void bias_grad_of(const Params& p, int h, double d, double* g0, double* g1, double* g2) {
    if (p.prior)
        bias_theta_grad(d, p.alpha[h], p.beta[h], p.mu[h], p.eps, g0, g1, g2);
    else
        bias_grad(d, p.alpha[h], p.beta[h], p.mu[h], p.eps, g0, g1, g2);
}

double dot(const double* a, const double* b, int D) {
    double acc = 0.0;
    for (int x = 0; x < D; ++x) acc += a[x] * b[x];
    return acc;
}

// Visible keys of query i: [0, i] causal, [0, T) otherwise.
int n_visible(int i, int T, int causal) { return causal ? (i + 1) : T; }

// Logit scale of query row i.
double row_scale(const Params& p, int h, int n, int D) {
    double inv = 1.0 / std::sqrt(static_cast<double>(D));
    if (p.ssmax) return p.s[h] * std::log(static_cast<double>(n)) * inv;
    return inv;
}

// One forward row: softmax over visible keys of z_ij, then the weighted sum of V.
// qi: the query row; kb, vb: the [T, D] keys and values of this (b, h);
// query position `pos` (distance d = pos - j); n visible keys 0..n-1.
void forward_row(const double* qi, const double* kb, const double* vb, int n,
                 int pos, int D, double c, const Params& p, int h, double* out, double* lse,
                 std::vector<double>& z) {
    z.resize(n);
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
        z[j] = c * dot(qi, kb + static_cast<size_t>(j) * D, D) +
               bias_of(p, h, static_cast<double>(pos - j));
        m = std::max(m, z[j]);
    }
    double l = 0.0;
    for (int x = 0; x < D; ++x) out[x] = 0.0;
    for (int j = 0; j < n; ++j) {
        double e = std::exp(z[j] - m);
        l += e;
        const double* vj = vb + static_cast<size_t>(j) * D;
        for (int x = 0; x < D; ++x) out[x] += e * vj[x];
    }
    for (int x = 0; x < D; ++x) out[x] /= l;
    *lse = m + std::log(l);
}

template <class F>
void parallel_for(int64_t n, int nthreads, F fn) {
    if (nthreads <= 0) nthreads = static_cast<int>(std::thread::hardware_concurrency());
    if (nthreads <= 0) nthreads = 1;
    nthreads = static_cast<int>(std::min<int64_t>(nthreads, std::max<int64_t>(n, 1)));
    std::atomic<int64_t> next(0);
    auto worker = [&]() {
        for (;;) {
            int64_t t = next.fetch_add(1);
            if (t >= n) break;
            fn(t);
        }
    };
    if (nthreads == 1) {
        worker();
        return;
    }
    std::vector<std::thread> pool;
    for (int t = 0; t < nthreads; ++t) pool.emplace_back(worker);
    for (auto& th : pool) th.join();
}

}  // namespace

extern "C" {

// b(d) for one head; exposed so that tests can check the bias in isolation.
// prior 1: (alpha, beta, mu) are (theta_alpha, theta_beta, theta_mu).
double bam_oracle_bias(double d, double alpha, double beta, double mu, double eps, int prior) {
    return prior ? bias_theta(d, alpha, beta, mu, eps) : bias(d, alpha, beta, mu, eps);
}

// The three partials of b at distance d; out[3].
void bam_oracle_bias_grad(double d, double alpha, double beta, double mu, double eps,
                          int prior, double* out) {
    if (prior)
        bias_theta_grad(d, alpha, beta, mu, eps, out, out + 1, out + 2);
    else
        bias_grad(d, alpha, beta, mu, eps, out, out + 1, out + 2);
}

// Forward of selected rows.  rows[r] = (b*H + h)*T + i.  o: [nrows, D], lse: [nrows].
int bam_oracle_fwd_rows(const double* q, const double* k, const double* v, int B, int H,
                        int T, int D, const double* alpha, const double* beta,
                        const double* mu, const double* s, double eps, int causal,
                        int ssmax, int prior, const int64_t* rows, int64_t nrows, double* o,
                        double* lse, int nthreads) {
    if (B < 1 || H < 1 || T < 1 || D < 1) return 1;
    Params p{alpha, beta, mu, s, eps, causal, ssmax, prior};
    parallel_for(nrows, nthreads, [&](int64_t r) {
        thread_local std::vector<double> z;
        int64_t flat = rows[r];
        int i = static_cast<int>(flat % T);
        int64_t bh = flat / T;
        int h = static_cast<int>(bh % H);
        size_t base = static_cast<size_t>(bh) * T * D;
        int n = n_visible(i, T, causal);
        double c = row_scale(p, h, n, D);
        forward_row(q + base + static_cast<size_t>(i) * D, k + base, v + base, n, i, D, c,
                    p, h, o + static_cast<size_t>(r) * D, lse + r, z);
    });
    return 0;
}

// Full forward: o [B,H,T,D], lse [B,H,T].
int bam_oracle_fwd(const double* q, const double* k, const double* v, int B, int H, int T,
                   int D, const double* alpha, const double* beta, const double* mu,
                   const double* s, double eps, int causal, int ssmax, int prior, double* o,
                   double* lse, int nthreads) {
    if (B < 1 || H < 1 || T < 1 || D < 1) return 1;
    Params p{alpha, beta, mu, s, eps, causal, ssmax, prior};
    parallel_for(static_cast<int64_t>(B) * H * T, nthreads, [&](int64_t flat) {
        thread_local std::vector<double> z;
        int i = static_cast<int>(flat % T);
        int64_t bh = flat / T;
        int h = static_cast<int>(bh % H);
        size_t base = static_cast<size_t>(bh) * T * D;
        int n = n_visible(i, T, causal);
        double c = row_scale(p, h, n, D);
        forward_row(q + base + static_cast<size_t>(i) * D, k + base, v + base, n, i, D, c,
                    p, h, o + static_cast<size_t>(flat) * D, lse + flat, z);
    });
    return 0;
}

// Decode: one new query per (b, h) against a cache of Tkv keys that includes it.
// The query sits at position Tkv-1, every cached key is visible, n = Tkv.
// q: [B,H,D]; kc, vc: [B,H,Tkv,D]; o: [B,H,D]; lse: [B,H].
int bam_oracle_decode(const double* q, const double* kc, const double* vc, int B, int H,
                      int Tkv, int D, const double* alpha, const double* beta,
                      const double* mu, const double* s, double eps, int ssmax, int prior,
                      double* o, double* lse, int nthreads) {
    if (B < 1 || H < 1 || Tkv < 1 || D < 1) return 1;
    Params p{alpha, beta, mu, s, eps, 1, ssmax, prior};
    parallel_for(static_cast<int64_t>(B) * H, nthreads, [&](int64_t bh) {
        thread_local std::vector<double> z;
        int h = static_cast<int>(bh % H);
        size_t base = static_cast<size_t>(bh) * Tkv * D;
        double c = row_scale(p, h, Tkv, D);
        forward_row(q + static_cast<size_t>(bh) * D, kc + base, vc + base, Tkv, Tkv - 1, D,
                    c, p, h, o + static_cast<size_t>(bh) * D, lse + bh, z);
    });
    return 0;
}

// Backward of L = sum(O * dO) by the plain chain rule.
//   P_ij = softmax_j(z_ij),  dP_ij = dO_i . v_j,  Delta_i = sum_j P_ij dP_ij,
//   dS_ij = P_ij (dP_ij - Delta_i)                          (= dL/dz_ij)
//   dq_i = sum_j dS_ij c_i k_j,  dk_j = sum_i dS_ij c_i q_i,  dv_j = sum_i P_ij dO_i
//   dalpha_h = sum dS_ij db/dalpha(i-j), likewise dbeta_h and dmu_h,
//   ds_h = sum dS_ij ln(n_i) q_i.k_j / sqrt(D)   (0 without SSMax).
// grads: dalpha, dbeta, dmu, ds are [H] (summed over the batch).
// absg (may be NULL): [4, H] sums of |per-element term| for each scalar gradient,
// the scale against which a near-cancelling scalar gradient is judged.
// absp (may be NULL): [4, H] sums of P_ij (|dP_ij| + |Delta_i|) |X_ij|, the
// magnitudes before the cancellation inside dS = P (dP - Delta): the scale of
// the rounding noise that any fp32 evaluation of the same sum carries.
int bam_oracle_bwd(const double* q, const double* k, const double* v, const double* dO,
                   int B, int H, int T, int D, const double* alpha, const double* beta,
                   const double* mu, const double* s, double eps, int causal, int ssmax,
                   int prior, double* dq, double* dk, double* dv, double* dalpha,
                   double* dbeta, double* dmu, double* ds, double* absg, double* absp,
                   int nthreads) {
    if (B < 1 || H < 1 || T < 1 || D < 1) return 1;
    Params p{alpha, beta, mu, s, eps, causal, ssmax, prior};
    const int64_t BH = static_cast<int64_t>(B) * H;
    std::vector<double> part(static_cast<size_t>(BH) * 12, 0.0);
    const double invsqrt = 1.0 / std::sqrt(static_cast<double>(D));
    parallel_for(BH, nthreads, [&](int64_t bh) {
        int h = static_cast<int>(bh % H);
        size_t base = static_cast<size_t>(bh) * T * D;
        const double* qb = q + base;
        const double* kb = k + base;
        const double* vb = v + base;
        const double* gb = dO + base;
        double* dqb = dq + base;
        double* dkb = dk + base;
        double* dvb = dv + base;
        std::fill(dqb, dqb + static_cast<size_t>(T) * D, 0.0);
        std::fill(dkb, dkb + static_cast<size_t>(T) * D, 0.0);
        std::fill(dvb, dvb + static_cast<size_t>(T) * D, 0.0);
        std::vector<double> z(T), P(T), dP(T);
        double acc[4] = {0, 0, 0, 0}, aabs[4] = {0, 0, 0, 0}, apre[4] = {0, 0, 0, 0};
        for (int i = 0; i < T; ++i) {
            int n = n_visible(i, T, causal);
            double c = row_scale(p, h, n, D);
            const double* qi = qb + static_cast<size_t>(i) * D;
            const double* gi = gb + static_cast<size_t>(i) * D;
            double m = -INFINITY;
            for (int j = 0; j < n; ++j) {
                z[j] = c * dot(qi, kb + static_cast<size_t>(j) * D, D) +
                       bias_of(p, h, static_cast<double>(i - j));
                m = std::max(m, z[j]);
            }
            double l = 0.0;
            for (int j = 0; j < n; ++j) {
                P[j] = std::exp(z[j] - m);
                l += P[j];
            }
            double delta = 0.0;
            for (int j = 0; j < n; ++j) {
                P[j] /= l;
                dP[j] = dot(gi, vb + static_cast<size_t>(j) * D, D);
                delta += P[j] * dP[j];
            }
            for (int j = 0; j < n; ++j) {
                double dS = P[j] * (dP[j] - delta);
                const double* kj = kb + static_cast<size_t>(j) * D;
                double* dkj = dkb + static_cast<size_t>(j) * D;
                double* dvj = dvb + static_cast<size_t>(j) * D;
                double* dqi = dqb + static_cast<size_t>(i) * D;
                for (int x = 0; x < D; ++x) {
                    dqi[x] += dS * c * kj[x];
                    dkj[x] += dS * c * qi[x];
                    dvj[x] += P[j] * gi[x];
                }
                double ga, gbeta, gm;
                bias_grad_of(p, h, static_cast<double>(i - j), &ga, &gbeta, &gm);
                double gs = ssmax ? std::log(static_cast<double>(n)) * invsqrt * dot(qi, kj, D)
                                  : 0.0;
                double t[4] = {dS * ga, dS * gbeta, dS * gm, dS * gs};
                double x[4] = {ga, gbeta, gm, gs};
                const double pre = P[j] * (std::fabs(dP[j]) + std::fabs(delta));
                for (int w = 0; w < 4; ++w) {
                    acc[w] += t[w];
                    aabs[w] += std::fabs(t[w]);
                    apre[w] += pre * std::fabs(x[w]);
                }
            }
        }
        for (int w = 0; w < 4; ++w) {
            part[static_cast<size_t>(bh) * 12 + w] = acc[w];
            part[static_cast<size_t>(bh) * 12 + 4 + w] = aabs[w];
            part[static_cast<size_t>(bh) * 12 + 8 + w] = apre[w];
        }
    });
    double* outs[4] = {dalpha, dbeta, dmu, ds};
    for (int w = 0; w < 4; ++w)
        for (int h = 0; h < H; ++h) outs[w][h] = 0.0;
    if (absg)
        for (int w = 0; w < 4 * H; ++w) absg[w] = 0.0;
    if (absp)
        for (int w = 0; w < 4 * H; ++w) absp[w] = 0.0;
    for (int64_t bh = 0; bh < BH; ++bh) {
        int h = static_cast<int>(bh % H);
        for (int w = 0; w < 4; ++w) {
            outs[w][h] += part[static_cast<size_t>(bh) * 12 + w];
            if (absg) absg[w * H + h] += part[static_cast<size_t>(bh) * 12 + 4 + w];
            if (absp) absp[w * H + h] += part[static_cast<size_t>(bh) * 12 + 8 + w];
        }
    }
    return 0;
}

}  // extern "C"
