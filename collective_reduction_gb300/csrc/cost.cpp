// Step-form cost model and schedule selection ("A Generalization of the
// Allreduce Operation", eqs. 36-37).  Host only; uses the public schedule
// compiler for the counters of each candidate.
#include <cmath>
#include <limits>
#include <vector>

#include "ar.h"
#include "schedule.hpp"

namespace {

// Fitted on GB300 by `bench.py --costmodel`: non-negative least squares on
// relative error over 126 step-form plans (ring, binomial, RD, generalized
// r = 0 and r = L, the ring's two halves; P = 4, 16, 63; 2 KiB .. 64 MiB per
// rank), rms relative error 0.24, with the kernels launched as programmatic
// dependents.  A combined byte costs a fifth of a sent one (the receiver's
// extra read mostly hides under the message), a message about 5 ns on top
// of its bytes: what makes thousands of tiny transfers expensive.
constexpr ar_cost_model kGB300 = {3.09, 3.00e-7, 7.10e-8, 4.81e-3};

bool model_ok(const ar_cost_model* m) {
    return m && m->alpha_us > 0 && m->beta_us_per_byte >= 0 && m->gamma_us_per_byte >= 0 &&
           m->delta_us_per_message >= 0 && std::isfinite(m->alpha_us) && std::isfinite(m->beta_us_per_byte) &&
           std::isfinite(m->gamma_us_per_byte) && std::isfinite(m->delta_us_per_message);
}

// Eq. (36) in the engine's terms: with u = m / P bytes per chunk and the
// per-process costs beta_p = P beta, gamma_p = P gamma,
//   T(r) = (2L - r) alpha + 2 (P - 1) m beta + (P - 1) m gamma
//          + (2^r - 1) L m beta + (2^r - 1) (2L - 2) m gamma,   0 <= r < L.
double eq36(int P, int L, double m, const ar_cost_model& c, int r) {
    const double e = std::ldexp(1.0, r) - 1.0;
    return (2.0 * L - r) * c.alpha_us + 2.0 * (P - 1) * m * c.beta_us_per_byte +
           (P - 1) * m * c.gamma_us_per_byte + e * L * m * c.beta_us_per_byte +
           e * (2.0 * L - 2.0) * m * c.gamma_us_per_byte;
}

}  // namespace

extern "C" {

ar_status ar_cost_model_default(ar_cost_model* out) {
    if (!out) return AR_ERR_INVALID_ARG;
    *out = kGB300;
    return AR_OK;
}

ar_status ar_cost_predict(ar_schedule_t s, const ar_cost_model* model, double* us) {
    if (!s || !model_ok(model) || !us) return AR_ERR_INVALID_ARG;
    ar_plan_info i;
    const ar_status st = ar_schedule_query(s, &i);
    if (st != AR_OK) return st;
    const double combined = static_cast<double>(i.combines) * ar::esize_of(i.dtype);
    *us = model->alpha_us * i.steps + model->beta_us_per_byte * static_cast<double>(i.sent_bytes_total) +
          model->gamma_us_per_byte * combined + model->delta_us_per_message * static_cast<double>(i.messages);
    return AR_OK;
}

ar_status ar_cost_optimal_r(int P, uint64_t bytes_per_rank, const ar_cost_model* model, int* r) {
    if (P < 1 || P > AR_MAX_RANKS || bytes_per_rank == 0 || !model_ok(model) || !r) return AR_ERR_INVALID_ARG;
    const int L = ar::ceil_log2(P);
    if (L <= 1) {  // only r = 0 lies below L
        *r = 0;
        return AR_OK;
    }
    const double m = static_cast<double>(bytes_per_rank);
    const double slope = std::log(2.0) * m * (L * model->beta_us_per_byte + (2.0 * L - 2.0) * model->gamma_us_per_byte);
    // eq. (37); a free byte (slope 0) pushes r* to the top of the range
    const double rs = slope > 0 ? std::log2(model->alpha_us / slope) : std::numeric_limits<double>::infinity();
    int lo = 0, hi = 0;
    if (rs >= L - 1) {
        lo = hi = L - 1;
    } else if (rs <= 0) {
        lo = hi = 0;
    } else {
        lo = static_cast<int>(std::floor(rs));
        hi = lo + 1 > L - 1 ? L - 1 : lo + 1;
    }
    *r = eq36(P, L, m, *model, hi) < eq36(P, L, m, *model, lo) ? hi : lo;
    return AR_OK;
}

ar_status ar_cost_select(int P, uint64_t n, ar_dtype dtype, ar_op op, const ar_cost_model* model,
                         ar_algo* algo, ar_params* params, double* us) {
    if (!model_ok(model) || !algo || !params || !us) return AR_ERR_INVALID_ARG;
    if (P < 1) return AR_ERR_INVALID_ARG;
    if (P > AR_MAX_RANKS) return AR_ERR_UNSUPPORTED;
    struct Cand {
        ar_algo algo;
        int r, k1;
    };
    std::vector<Cand> cands{{AR_RING, 0, 0}, {AR_BINOMIAL, 0, 0}, {AR_RD, 0, 0}, {AR_RH, 0, 0}};
    int Lp = 0;
    while ((2 << Lp) <= P) ++Lp;  // log2 of the largest power of two <= P
    for (int k1 = 0; k1 <= Lp; ++k1) cands.push_back({AR_HYBRID, 0, k1});
    for (int r = 0; r <= ar::ceil_log2(P); ++r) cands.push_back({AR_GENERALIZED, r, 0});
    double best = std::numeric_limits<double>::infinity();
    bool found = false;
    for (const Cand& c : cands) {
        ar_params p{};
        p.form = AR_FORM_STEP;
        p.order = AR_ORDER_FAITHFUL;
        p.group = AR_GROUP_CYCLIC;
        p.r = c.r;
        p.k1 = c.k1;
        p.blocks = 1;
        p.phase = AR_PHASE_ALLREDUCE;
        ar_schedule_t s = nullptr;
        const ar_status st = ar_schedule_create(P, n, dtype, op, c.algo, &p, &s);
        if (st != AR_OK) return st;
        double t = 0;
        const ar_status pt = ar_cost_predict(s, model, &t);
        ar_schedule_destroy(s);
        if (pt != AR_OK) return pt;
        if (t < best) {
            best = t;
            *algo = c.algo;
            *params = p;
            found = true;
        }
    }
    if (!found) return AR_ERR_INVALID_ARG;
    *us = best;
    return AR_OK;
}

}  // extern "C"
