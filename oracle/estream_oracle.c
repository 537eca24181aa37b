/*
 * estream_oracle.c -- plain CPU oracle for one MoE layer's prefill.
 *
 * TEST INFRASTRUCTURE. This is the slow, obviously correct restatement of what
 * the method computes, used only by the tests, by smoke() and by the bench's
 * CPU-baseline leg. The CUDA library never links, loads or calls it, and it
 * shares no code, header, table or constant with the CUDA sources.
 *
 * Source: "EStream: Fast and Memory-Efficient MoE Prefill through Expert
 * Virtualization on Mobile NPUs" (arXiv 2609.06551).
 *   - Eq. 1 (section 3.2): F_e(X_t) = W_e^d ( SiLU(W_e^g X_t) (*) W_e^u X_t ).
 *   - Eq. 2 (section 3.2): Y_t = A_t + sum over (e, alpha) in R_l(t) of alpha * F_e(X_t).
 *   - Section 3.2, "Composed Sparse Route and Parameter Binding", and the
 *     route-map part of Algorithm 1: slot resolution psi_i = Phi_l(e_i),
 *     per-slot counts, exclusive prefix sum, and a second pass that stores
 *     (t_i, i) contiguously by slot.
 *   - Eq. 4 (section 3.3): grouped placement Phi_l(e) = b*G + (pi_l(e) mod G)
 *     when group floor(pi_l(e)/G) resides in bank b.
 *
 * Readings where the pages are silent (each is listed in the design notes):
 *   - Router scores are a softmax over the E logits (the pages say only
 *     "top-k of E experts"). Top-k order: larger logit first, equal logits ->
 *     lower expert id first. Route index i = t*k + j (token-major, rank-minor).
 *   - alpha = softmax probability p, or p / (sum of the k selected p, summed in
 *     rank order) when renormalisation is asked for.
 *   - Routing arithmetic is fp32 with one written exponential (below); the
 *     expert FFN is evaluated in fp64 from the fp32/bf16 inputs widened exactly.
 *   - Routes whose slot is "not resident" (Phi = -1) go to a trailing bucket P,
 *     so the CSR always holds all R = T*k routes; offsets has P+2 entries.
 *
 * The written exponential (fp32; the same written definition is implemented
 * independently by the CUDA routing kernel so that alpha is bit-exact):
 *   for x < -87: 0
 *   n = round-half-even( fl(x * LOG2E) )
 *   r = fma(-n, LN2_HI, x);  r = fma(-n, LN2_LO, r)     Cody & Waite (1980)
 *   p = Horner form of sum_{j=0..7} r^j / j!, one fma per step
 *   exp(x) = p * 2^n                                      (exact scaling)
 * LN2_HI is ln 2 rounded to fp32 with its 8 low significand bits cleared (so
 * n * LN2_HI is exact for |n| < 256); LN2_LO = fp32(ln 2 - LN2_HI); LOG2E and
 * the 1/j! are the round-to-nearest fp32 values of 1/ln 2 and 1/j!.
 * Compile with -ffp-contract=off: every rounding step is written out.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Written exponential                                                       */
/* ------------------------------------------------------------------------ */

static const float O_LOG2E = 0x1.715476p+0f;   /* fp32(1/ln 2) */
static const float O_LN2_HI = 0x1.62e4p-1f;    /* ln 2 to 16 significant bits */
static const float O_LN2_LO = 0x1.7f7d1cp-20f; /* fp32(ln 2 - O_LN2_HI) */

float oracle_exp_f32(float x)
{
    if (x < -87.0f) return 0.0f;
    float t = x * O_LOG2E;
    float n = nearbyintf(t);              /* default rounding mode: half to even */
    float r = fmaf(-n, O_LN2_HI, x);
    r = fmaf(-n, O_LN2_LO, r);
    /* 1/j! for j = 7..0, fp32 round-to-nearest */
    float p = 0x1.a01a02p-13f;            /* 1/5040 */
    p = fmaf(p, r, 0x1.6c16c2p-10f);      /* 1/720 */
    p = fmaf(p, r, 0x1.111112p-7f);       /* 1/120 */
    p = fmaf(p, r, 0x1.555556p-5f);       /* 1/24 */
    p = fmaf(p, r, 0x1.555556p-3f);       /* 1/6 */
    p = fmaf(p, r, 0.5f);                 /* 1/2 */
    p = fmaf(p, r, 1.0f);                 /* 1/1 */
    p = fmaf(p, r, 1.0f);                 /* 1/0! */
    int ni = (int)n;                      /* in [-126, 0] for x in [-87, 0] */
    union { uint32_t u; float f; } scale;
    scale.u = (uint32_t)(ni + 127) << 23;
    return p * scale.f;
}

/* ------------------------------------------------------------------------ */
/* Router: softmax top-k                                                     */
/* ------------------------------------------------------------------------ */

/* For every token t: ids of the k largest logits (ties -> lower id first) and
 * their routing weights. Returns 0, or -1 on bad arguments. */
int oracle_route_topk(const float* logits, int T, int E, int k, int renorm,
                      int32_t* topk_ids, float* alpha)
{
    if (T < 0 || E < 1 || k < 1 || k > E) return -1;
    float* prob = (float*)malloc(sizeof(float) * (size_t)E);
    unsigned char* taken = (unsigned char*)malloc((size_t)E);
    if (!prob || !taken) { free(prob); free(taken); return -1; }
    for (int t = 0; t < T; ++t) {
        const float* l = logits + (size_t)t * E;
        /* softmax: subtract the maximum, exponentiate, sum in ascending e */
        float m = l[0];
        for (int e = 1; e < E; ++e) if (l[e] > m) m = l[e];
        float s = 0.0f;
        for (int e = 0; e < E; ++e) {
            prob[e] = oracle_exp_f32(l[e] - m);
            s = s + prob[e];
        }
        for (int e = 0; e < E; ++e) prob[e] = prob[e] / s;
        /* selection: k passes, each taking the largest remaining logit */
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || l[e] > l[best]) best = e;   /* strict: ties keep the lower id */
            }
            taken[best] = 1;
            topk_ids[(size_t)t * k + j] = best;
            alpha[(size_t)t * k + j] = prob[best];
        }
        if (renorm) {
            float z = 0.0f;
            for (int j = 0; j < k; ++j) z = z + alpha[(size_t)t * k + j];
            for (int j = 0; j < k; ++j) alpha[(size_t)t * k + j] = alpha[(size_t)t * k + j] / z;
        }
    }
    free(prob);
    free(taken);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Route map (CSR by physical slot)                                          */
/* ------------------------------------------------------------------------ */

/* Composed route binding of section 3.2 / Algorithm 1 (route-map part).
 * Route i = t*k + j goes to logical expert e_i = topk_ids[i]. Its slot is
 * psi_i = phi[e_i] (phi == NULL means the identity, which needs P == E);
 * phi[e] == -1 means "not resident", which this restatement files under the
 * trailing bucket P. Outputs:
 *   offsets[0..P+1]: offsets[0] = 0, offsets[s+1] = offsets[s] + count[s]
 *   rec_tok[p], rec_route[p]: the record (t_i, i) at position p.
 * Returns 0, or -1 on bad arguments (an id or slot out of range). */
int oracle_route_csr(const int32_t* topk_ids, int T, int k, const int32_t* phi,
                     int E, int P, int32_t* offsets, int32_t* rec_tok,
                     int32_t* rec_route)
{
    if (T < 0 || k < 1 || E < 1 || P < 0) return -1;
    if (!phi && P != E) return -1;
    const int R = T * k;
    int32_t* psi = (int32_t*)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    int32_t* count = (int32_t*)calloc((size_t)P + 1, sizeof(int32_t));
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * ((size_t)P + 2));
    if (!psi || !count || !cursor) { free(psi); free(count); free(cursor); return -1; }
    int rc = 0;
    /* resolve the physical slot of every route */
    for (int i = 0; i < R; ++i) {
        int e = topk_ids[i];
        if (e < 0 || e >= E) { rc = -1; break; }
        int s = phi ? phi[e] : e;
        if (s < -1 || s >= P) { rc = -1; break; }
        psi[i] = (s < 0) ? P : s;
    }
    if (rc == 0) {
        /* count routes per slot */
        for (int i = 0; i < R; ++i) count[psi[i]] += 1;
        /* exclusive prefix sum */
        offsets[0] = 0;
        for (int s = 0; s <= P; ++s) offsets[s + 1] = offsets[s] + count[s];
        /* second pass: store (t_i, i) contiguously by slot, in ascending i */
        for (int s = 0; s <= P; ++s) cursor[s] = offsets[s];
        for (int i = 0; i < R; ++i) {
            int p = cursor[psi[i]];
            rec_tok[p] = i / k;
            rec_route[p] = i;
            cursor[psi[i]] = p + 1;
        }
    }
    free(psi);
    free(count);
    free(cursor);
    return rc;
}

/* Eq. 4: placement of grouped experts. perm[e] = pi(e) (storage position),
 * bank_of_group[q] = the bank holding storage group q, or -1. Writes
 * phi[e] = b*G + (pi(e) mod G) when group floor(pi(e)/G) is in bank b, else -1. */
int oracle_grouped_placement(const int32_t* perm, int E, int G,
                             const int32_t* bank_of_group, int32_t* phi)
{
    if (E < 1 || G < 1) return -1;
    for (int e = 0; e < E; ++e) {
        int pos = perm ? perm[e] : e;
        if (pos < 0 || pos >= E) return -1;
        int q = pos / G;          /* storage group */
        int r = pos % G;          /* position inside the group */
        int b = bank_of_group[q];
        phi[e] = (b < 0) ? -1 : b * G + r;
    }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Expert FFN and layer output                                               */
/* ------------------------------------------------------------------------ */

/* Element access for the two input encodings: fp32, or bf16 bit patterns
 * (the upper 16 bits of an fp32), both widened exactly to double. */
static double load_elem(const void* base, size_t idx, int bf16)
{
    if (bf16) {
        union { uint32_t u; float f; } v;
        v.u = (uint32_t)((const uint16_t*)base)[idx] << 16;
        return (double)v.f;
    }
    return (double)((const float*)base)[idx];
}

static double silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------------ */
/* 4-bit expert weights (weight-only Q4_0-style block quantisation)          */
/* ------------------------------------------------------------------------ */

/* Section 4 ("Numerical representation") stores expert matrices as weight-only
 * GGUF Q4_0: blocks of 32 consecutive weights along the reduction dimension,
 * one scale per block, a 4-bit code per weight with offset 8. Reading used
 * here (the pages give only the format's name):
 *   m   = the block's element of largest magnitude (the first one on ties);
 *   d   = m / -8, rounded to 5 significant bits (round to nearest, ties to
 *         even), then to the matrix-operand type (bf16, or fp16 when fp16 is
 *         set) -- with at most 5 significant bits in d, every (q - 8) * d is
 *         exact in either type;
 *   q_j = clamp(rint(x_j / d) + 8, 0, 15)   (fp32 division, ties to even);
 *   a block of zeros has d = 0 and every q_j = 8.
 * The weight the layer uses is w_j = (q_j - 8) * d. For a down plane the
 * weights are first multiplied by 2^s, s = 15 - e where the plane's largest
 * magnitude is f * 2^e with f in [0.5, 1) (s = 0 for an all-zero plane), and
 * the dequantised weight is divided by 2^s again. */

static float round_sig5(float x)
{
    union { float f; uint32_t u; } v;
    v.f = x;
    const uint32_t drop = 19;                    /* keep 1 implicit + 4 stored bits */
    const uint32_t half = 1u << (drop - 1);
    const uint32_t lsb = (v.u >> drop) & 1u;
    v.u = (v.u + half - 1u + lsb) & ~((1u << drop) - 1u);
    return v.f;
}

static float to_bf16_rne(float x)
{
    union { float f; uint32_t u; } v;
    v.f = x;
    v.u = (v.u + 0x7FFFu + ((v.u >> 16) & 1u)) & 0xFFFF0000u;
    return v.f;
}

/* fp16 round to nearest even, returned as the fp32 of the fp16 value
 * (finite inputs below 65520 in magnitude). */
static float to_fp16_rne(float x)
{
    const double ax = fabs((double)x);
    if (ax == 0.0) return x;
    int e;
    frexp(ax, &e);                      /* ax = f * 2^e, f in [0.5, 1) */
    int q = e - 11;                     /* quantum of an 11-bit significand */
    if (q < -24) q = -24;               /* subnormal range: fixed quantum 2^-24 */
    const double scaled = ldexp(ax, -q);
    double r = nearbyint(scaled);       /* default rounding mode: ties to even */
    const double out = ldexp(r, q);
    return (float)(x < 0 ? -out : out);
}

int oracle_down_scale_exp(const void* w, size_t n, int bf16)
{
    double mx = 0.0;
    for (size_t i = 0; i < n; ++i) {
        const double a = fabs(load_elem(w, i, bf16));
        if (a > mx) mx = a;
    }
    if (mx == 0.0) return 0;
    int e;
    frexp(mx, &e);
    return 15 - e;
}

/* Quantise a [rows][cols] matrix (cols % 32 == 0) row by row along cols.
 * codes: [rows][cols] bytes 0..15; d: [rows][cols/32] fp32 (the stored scale,
 * widened exactly); scale_exp s multiplies the weights by 2^s first. */
int oracle_q4_quantize(const void* w, int rows, int cols, int bf16, int scale_exp, int fp16,
                       uint8_t* codes, float* d)
{
    if (rows < 0 || cols < 32 || cols % 32 != 0 || !w || !codes || !d) return -1;
    const int nb = cols / 32;
    for (int r = 0; r < rows; ++r)
        for (int b = 0; b < nb; ++b) {
            float x[32];
            float m = 0.0f;
            for (int j = 0; j < 32; ++j) {
                x[j] = (float)ldexp(load_elem(w, (size_t)r * cols + (size_t)b * 32 + j, bf16), scale_exp);
                if (fabsf(x[j]) > fabsf(m)) m = x[j];
            }
            float dd = 0.0f;
            if (m != 0.0f) {
                dd = round_sig5(m / -8.0f);
                dd = fp16 ? to_fp16_rne(dd) : to_bf16_rne(dd);
            }
            d[(size_t)r * nb + b] = dd;
            for (int j = 0; j < 32; ++j) {
                int q = 8;
                if (dd != 0.0f) {
                    q = (int)rintf(x[j] / dd) + 8;
                    if (q < 0) q = 0;
                    if (q > 15) q = 15;
                }
                codes[(size_t)r * cols + (size_t)b * 32 + j] = (uint8_t)q;
            }
        }
    return 0;
}

/* w[r][c] = (codes[r][c] - 8) * d[r][c/32] * 2^-scale_exp, in fp32 (exact). */
int oracle_q4_dequantize(const uint8_t* codes, const float* d, int rows, int cols, int scale_exp,
                         float* w)
{
    if (rows < 0 || cols < 32 || cols % 32 != 0 || !codes || !d || !w) return -1;
    const int nb = cols / 32;
    for (int r = 0; r < rows; ++r)
        for (int c = 0; c < cols; ++c)
            w[(size_t)r * cols + c] =
                (float)ldexp(((double)codes[(size_t)r * cols + c] - 8.0) * (double)d[(size_t)r * nb + c / 32],
                             -scale_exp);
    return 0;
}

/* Router logits upstream of the top-k (the layer input X_t mapped to one
 * score per expert; the pages name the router and its top-k selection in
 * section 1 and list a routing operator among the NPU operators in section 4,
 * without its form). Reading: the bias-free linear router of top-k MoE
 * layers, l[t][e] = sum over h of X[t][h] * W_r[e][h], evaluated in fp64 from
 * the exactly widened inputs (X [T][H], W_r [E][H], both fp32 or both bf16
 * bit patterns), ascending h. Returns 0, or -1 on bad arguments. */
int oracle_router_logits(const void* X, int T, int H, const void* W_r, int E, int bf16,
                         double* logits)
{
    if (T < 0 || H < 1 || E < 1 || (T > 0 && (!X || !W_r || !logits))) return -1;
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += load_elem(X, (size_t)t * H + h, bf16) * load_elem(W_r, (size_t)e * H + h, bf16);
            logits[(size_t)t * E + e] = acc;
        }
    return 0;
}

/* Eq. 1 for one token row: out[o] = sum_f Wd[o][f] * SiLU(g_f) * u_f with
 * g_f = sum_h Wg[f][h] x[h], u_f = sum_h Wu[f][h] x[h].
 * Wg, Wu are [F][H] and Wd is [H][F], row-major; x is the token's row offset
 * into X. hbuf is caller scratch of F doubles. */
static void expert_ffn_row(const void* X, size_t x_off, const void* Wg,
                           const void* Wu, const void* Wd, size_t w_off_gu,
                           size_t w_off_d, int H, int F, int bf16,
                           double* hbuf, double* out)
{
    for (int f = 0; f < F; ++f) {
        double g = 0.0, u = 0.0;
        for (int h = 0; h < H; ++h) {
            double xv = load_elem(X, x_off + (size_t)h, bf16);
            g += load_elem(Wg, w_off_gu + (size_t)f * H + h, bf16) * xv;
            u += load_elem(Wu, w_off_gu + (size_t)f * H + h, bf16) * xv;
        }
        hbuf[f] = silu(g) * u;
    }
    for (int o = 0; o < H; ++o) {
        double y = 0.0;
        for (int f = 0; f < F; ++f)
            y += load_elem(Wd, w_off_d + (size_t)o * F + f, bf16) * hbuf[f];
        out[o] = y;
    }
}

/* Eq. 2 for the tokens listed in rows[0..n_rows): for list entry r, token
 * t = rows[r],
 *   Y_out[r][:] = A_t + sum_j alpha[t*k+j] * F_{topk_ids[t*k+j]}(X_t)
 *                 + sum_{s < n_shared} F^shared_s(X_t)
 * Routed weights: Wg, Wu [E][F][H], Wd [E][H][F]. Shared experts (weight 1):
 * Sg, Su [n_shared][Fs][H], Sd [n_shared][H][Fs] (NULL when n_shared == 0).
 * X is [T][H]; A is the residual [T][H] in double, or NULL for zero.
 * bf16 != 0: X and every weight are bf16 bit patterns; else fp32. */
int oracle_moe_layer_rows(const void* X, int T, int H, int E, int F, int k,
                          const void* Wg, const void* Wu, const void* Wd,
                          const int32_t* topk_ids, const float* alpha,
                          int n_shared, int Fs, const void* Sg, const void* Su,
                          const void* Sd, const double* A, int bf16,
                          const int32_t* rows, int n_rows, double* Y_out)
{
    if (T < 0 || H < 1 || E < 1 || F < 1 || k < 1 || k > E || n_rows < 0) return -1;
    if (n_shared > 0 && (Fs < 1 || !Sg || !Su || !Sd)) return -1;
    for (int r = 0; r < n_rows; ++r)
        if (rows[r] < 0 || rows[r] >= T) return -1;
    for (int r = 0; r < n_rows; ++r)
        for (int j = 0; j < k; ++j) {
            int e = topk_ids[(size_t)rows[r] * k + j];
            if (e < 0 || e >= E) return -1;
        }
    int Fmax = F > Fs ? F : Fs;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int r = 0; r < n_rows; ++r) {
        double* hbuf = (double*)malloc(sizeof(double) * (size_t)Fmax);
        double* fo = (double*)malloc(sizeof(double) * (size_t)H);
        if (!hbuf || !fo) {
            free(hbuf);
            free(fo);
#pragma omp atomic write
            bad = 1;
            continue;
        }
        int t = rows[r];
        double* y = Y_out + (size_t)r * H;
        for (int o = 0; o < H; ++o) y[o] = A ? A[(size_t)t * H + o] : 0.0;
        size_t x_off = (size_t)t * H;
        for (int j = 0; j < k; ++j) {
            int e = topk_ids[(size_t)t * k + j];
            double a = (double)alpha[(size_t)t * k + j];
            expert_ffn_row(X, x_off, Wg, Wu, Wd, (size_t)e * F * H,
                           (size_t)e * H * F, H, F, bf16, hbuf, fo);
            for (int o = 0; o < H; ++o) y[o] += a * fo[o];
        }
        for (int s = 0; s < n_shared; ++s) {
            expert_ffn_row(X, x_off, Sg, Su, Sd, (size_t)s * Fs * H,
                           (size_t)s * H * Fs, H, Fs, bf16, hbuf, fo);
            for (int o = 0; o < H; ++o) y[o] += fo[o];
        }
        free(hbuf);
        free(fo);
    }
    return bad ? -1 : 0;
}

/* Number of threads the layer oracle runs on (1 without OpenMP). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ------------------------------------------------------------------------ */
/* Pipeline model                                                            */
/* ------------------------------------------------------------------------ */

/* Max-plus recurrence of the UFS-NPU pipeline (section 3.4, Eq. 5), for K
 * scheduled groups with read times L[k] and execution times X[k]
 * (k = 1..K stored at index k-1), queue depth q, bank count b and
 * non-expert completion T_ne:
 *   a_k = max(d_{k-q}, f_{k-b})      (a read waits for a queue slot and a free bank)
 *   d_k = a_k + L_k
 *   s_k = max(d_k, T_ne, f_{k-1})    (execution waits for its data, the
 *                                     non-expert work and the previous group)
 *   f_k = s_k + X_k
 * with d_j = f_j = 0 for j <= 0. Writes (a, d, s, f) per group into adsf if
 * not NULL and returns T_pipe = f_K. */
double oracle_maxplus(const double* L, const double* X, int K, int q, int b, double T_ne,
                      double* adsf)
{
    if (K <= 0) return T_ne > 0.0 ? T_ne : 0.0;
    double* d = (double*)calloc((size_t)K + 1, sizeof(double));
    double* f = (double*)calloc((size_t)K + 1, sizeof(double));
    if (!d || !f) { free(d); free(f); return -1.0; }
    for (int k = 1; k <= K; ++k) {
        double dq = (k - q >= 1) ? d[k - q] : 0.0;
        double fb = (k - b >= 1) ? f[k - b] : 0.0;
        double a = dq > fb ? dq : fb;
        d[k] = a + L[k - 1];
        double s = d[k];
        if (T_ne > s) s = T_ne;
        if (f[k - 1] > s) s = f[k - 1];   /* f[0] = 0 */
        f[k] = s + X[k - 1];
        if (adsf) {
            adsf[4 * (k - 1) + 0] = a;
            adsf[4 * (k - 1) + 1] = d[k];
            adsf[4 * (k - 1) + 2] = s;
            adsf[4 * (k - 1) + 3] = f[k];
        }
    }
    double out = f[K];
    free(d);
    free(f);
    return out;
}
