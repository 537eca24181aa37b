// Host-side pipeline model and automatic configuration of the expert arena.
//
// "EStream: Fast and Memory-Efficient MoE Prefill through Expert
// Virtualization on Mobile NPUs", section 3.4 ("Automatic Pipeline
// Configuration"):
//   Eq. 5  max-plus recurrence over the K scheduled groups of one layer:
//          a_k = max(d_{k-q}, f_{k-b}), d_k = a_k + L_k,
//          s_k = max(d_k, T_ne, f_{k-1}), f_k = s_k + X_k,
//          d_j = f_j = 0 for j <= 0, T_pipe = f_K;
//          L_k is group k's read time, X_k its execution time, q the number
//          of reads in flight, b the number of banks, T_ne the completion of
//          the layer's non-expert work.
//   Eq. 8  B_max(g) = min(floor((M_max - M_other(g)) / (g * W_e)), ceil(N_e / g))
//   Eq. 9  B*(g) = argmin over Q0 <= b <= B_max(g) of T_pipe(g, Q0, b)
//   Eq. 10 G* = argmin over g with B_max(g) >= Q0 of T_pipe(g, Q0, B*(g))
// (Eq. 6 is the joint problem Eqs. 7-10 decompose; Eq. 7 fixes Q0 from a
// measured bandwidth-vs-queue-depth sweep and is applied by the caller.)
// The calibration inputs (L_k, X_k per candidate g) come from one profiled
// layer call per g: estream_pipeline_trace records, per group, when its read
// started and ended and when its execution started and ended.
#include <algorithm>
#include <cmath>
#include <vector>

#include "estream_internal.h"

extern "C" double estream_maxplus_pipeline(const double* L, const double* X, int K, int q, int b,
                                           double T_ne, double* adsf) {
    if (K <= 0) return T_ne > 0.0 ? T_ne : 0.0;
    if (!L || !X || q < 1 || b < 1) return -1.0;
    std::vector<double> d(static_cast<size_t>(K) + 1, 0.0), f(static_cast<size_t>(K) + 1, 0.0);
    // index k = 1..K; index 0 (and anything <= 0) reads as 0
    auto at = [](const std::vector<double>& v, int j) { return j <= 0 ? 0.0 : v[j]; };
    for (int k = 1; k <= K; ++k) {
        const double a = std::max(at(d, k - q), at(f, k - b));
        d[k] = a + L[k - 1];
        const double s = std::max(std::max(d[k], T_ne), at(f, k - 1));
        f[k] = s + X[k - 1];
        if (adsf) {
            adsf[4 * (k - 1) + 0] = a;
            adsf[4 * (k - 1) + 1] = d[k];
            adsf[4 * (k - 1) + 2] = s;
            adsf[4 * (k - 1) + 3] = f[k];
        }
    }
    return f[K];
}

extern "C" int estream_bank_bound(int g, double M_max, double M_other, double W_e, int N_e) {
    if (g < 1 || W_e <= 0.0 || N_e < 1) return 0;
    const double room = M_max - M_other;
    if (room <= 0.0) return 0;
    const long long by_mem = static_cast<long long>(std::floor(room / (g * W_e)));
    const long long groups = (static_cast<long long>(N_e) + g - 1) / g;
    return static_cast<int>(std::max(0ll, std::min(by_mem, groups)));
}

extern "C" estream_status estream_autoconfig(int n_g, const int* g_values, const int* K_per_g,
                                             const double* const* L_per_g,
                                             const double* const* X_per_g, double T_ne, int Q0,
                                             double M_max, const double* M_other_per_g,
                                             double W_e, int N_e, int* G_out, int* B_out,
                                             double* T_out) {
    if (n_g < 1 || !g_values || !K_per_g || !L_per_g || !X_per_g || Q0 < 1 || W_e <= 0.0 ||
        N_e < 1 || !G_out || !B_out)
        return ESTREAM_ERR_INVALID_ARG;
    int best_g = -1, best_b = -1;
    double best_t = 0.0;
    for (int i = 0; i < n_g; ++i) {
        const int g = g_values[i];
        const double m_other = M_other_per_g ? M_other_per_g[i] : 0.0;
        const int bmax = estream_bank_bound(g, M_max, m_other, W_e, N_e);
        if (bmax < Q0) continue;  // Eq. 10's feasibility condition
        int bstar = -1;
        double tstar = 0.0;
        for (int b = Q0; b <= bmax; ++b) {  // Eq. 9
            const double t = estream_maxplus_pipeline(L_per_g[i], X_per_g[i], K_per_g[i], Q0, b,
                                                      T_ne, nullptr);
            if (t < 0.0) return ESTREAM_ERR_INVALID_ARG;
            if (bstar < 0 || t < tstar) {  // strict: ties keep the smaller bank count
                bstar = b;
                tstar = t;
            }
        }
        if (best_g < 0 || tstar < best_t) {  // Eq. 10; ties keep the earlier candidate
            best_g = g;
            best_b = bstar;
            best_t = tstar;
        }
    }
    if (best_g < 0) return ESTREAM_ERR_CAPACITY;
    *G_out = best_g;
    *B_out = best_b;
    if (T_out) *T_out = best_t;
    return ESTREAM_OK;
}
