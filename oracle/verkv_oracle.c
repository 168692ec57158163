/*
 * VerKV oracle -- TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.
 *
 * A plain, slow, double-precision CPU restatement of the method in
 * "Verify Before You Fetch: Reliable KV Cache Compression for LLM Inference"
 * (PoissonComp, Algorithm 1 and Sec. 4.1, eq. (3); KVFetch, Algorithm 2 and
 * Sec. 4.2, Definition 2 / eq. (5), Theorem 1 / eq. (6), Lemma 1 / eq. (7),
 * eqs. (9)-(10), Theorem 2; binary shrinkage, Appendix A.2; key sketch and
 * shortlist, Appendix A.1).
 *
 * Only the test-suite, the package smoke check and the CPU-baseline leg of
 * the benchmark may load this library.  It shares no code with the CUDA
 * library: the two are written independently from the paper and compared.
 *
 * Build: gcc -O2 -ffp-contract=off -fopenmp -shared -fPIC (no fast-math; the
 * contraction switch matters on aarch64, where gcc fuses a*b+c by default).
 *
 * Conventions (readings of the paper where it is silent are listed here and
 * in the design notes):
 *   flags: 2 = H (kept with probability one), 1 = S (in L and sampled),
 *          0 = in L and not sampled.
 *   Importance scores tau are fp32 data.  Tokens of the sink/local windows
 *   are forced to tau = 1 (Algorithm 1, scoring step) and lie outside the
 *   water-filling; every other score is floored at 2^-38 so that every token
 *   is in H or L (the paper defines L by 0 < r_i < 1).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define VKO_TAU_FLOOR 0x1p-38f

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon, Moraes, Dror, Shaw: "Parallel random numbers: as   */
/* easy as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies, with    */
/* the key bumped by the Weyl constants between rounds.                      */
/* ------------------------------------------------------------------------ */
void vko_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4])
{
    const uint32_t mul0 = 0xD2511F53u, mul1 = 0xCD9E8D57u;
    const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)mul0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)mul1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        c0 = n0; c1 = lo1; c2 = n2; c3 = lo0;
        k0 += weyl0; k1 += weyl1;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Uniform draw for token `token` of KV head `kv_head` in layer `layer` of
 * sequence `seq`: word x of Philox4x32-10 at key (seed_lo, seed_hi) and
 * counter (token, kv_head, layer, seq); u = floor(x / 2^8) * 2^-24, an exact
 * fp32 value in [0, 1). */
float vko_uniform(uint64_t seed, uint32_t token, uint32_t kv_head, uint32_t layer, uint32_t seq)
{
    uint32_t ctr[4] = {token, kv_head, layer, seq};
    uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
    uint32_t out[4];
    vko_philox4x32_10(ctr, key, out);
    return (float)(out[0] >> 8) * 0x1p-24f;
}

/* ------------------------------------------------------------------------ */
/* Importance scores (Algorithm 1, scoring step).  The scorer C of the paper is a  */
/* trained model; the synthetic stand-in is: for every observation query row */
/* j, p_j = softmax over tokens of <Q_j, K_i>/sqrt(d); tau_i = max_j p_j(i), */
/* divided by its maximum over i; tau = 1 on the sink and local windows.     */
/* K: [n][d], Q: [rows][d] (doubles).  Output: fp32 tau with the floor.      */
/* ------------------------------------------------------------------------ */
void vko_tau(int64_t n, int d, const double* K, int rows, const double* Q,
             int n_sink, int n_local, float* tau_out)
{
    double* best = (double*)malloc(sizeof(double) * (size_t)n);
    double* logit = (double*)malloc(sizeof(double) * (size_t)n);
    const double inv_sqrt_d = 1.0 / sqrt((double)d);
    for (int64_t i = 0; i < n; ++i) best[i] = 0.0;
    for (int j = 0; j < rows; ++j) {
        double mx = -INFINITY;
        for (int64_t i = 0; i < n; ++i) {
            double s = 0.0;
            for (int c = 0; c < d; ++c) s += Q[(size_t)j * d + c] * K[(size_t)i * d + c];
            logit[i] = s * inv_sqrt_d;
            if (logit[i] > mx) mx = logit[i];
        }
        double z = 0.0;
        for (int64_t i = 0; i < n; ++i) z += exp(logit[i] - mx);
        for (int64_t i = 0; i < n; ++i) {
            double p = exp(logit[i] - mx) / z;
            if (p > best[i]) best[i] = p;
        }
    }
    double top = 0.0;
    for (int64_t i = 0; i < n; ++i) if (best[i] > top) top = best[i];
    for (int64_t i = 0; i < n; ++i) {
        float t = (float)(best[i] / top);
        if (t < VKO_TAU_FLOOR) t = VKO_TAU_FLOOR;
        if (i < n_sink || i >= n - n_local) t = 1.0f;
        tau_out[i] = t;
    }
    free(best);
    free(logit);
}

/* ------------------------------------------------------------------------ */
/* Water-filling (Algorithm 1, water-filling step; eq. (3)).                 */
/* I = sink/local tokens (always in H).  U = the rest, B' = budget - |I|.    */
/* Find c with sum_{i in U} min(1, c tau_i) = B' exactly as the paper's c:   */
/* sort U by tau descending; with the top t capped, c_t = (B' - t) / S_t,    */
/* S_t the sum of the remaining scores; the answer is the first t whose next */
/* score is below the cap, (B' - t) * tau_(t) < S_t (0-based, tau_(t) is the */
/* largest uncapped score).  S_t is summed exactly (scores >= 2^-38 are      */
/* integers in units of 2^-61) and rounded to double once.                  */
/* r_i = min(1, c tau_i) in double (r64) and rounded to fp32 (r32); the fp32 */
/* value is the stored inclusion probability and decides H = {r32 == 1}.     */
/* Returns 0, or -1 when B' <= 0 (budget does not cover the forced set).    */
/* ------------------------------------------------------------------------ */
static _Thread_local const float* g_sort_tau;   /* per thread: rows run in parallel */
static int cmp_tau_desc(const void* a, const void* b)
{
    int64_t ia = *(const int64_t*)a, ib = *(const int64_t*)b;
    float ta = g_sort_tau[ia], tb = g_sort_tau[ib];
    if (ta > tb) return -1;
    if (ta < tb) return 1;
    return (ia < ib) ? -1 : (ia > ib);
}

static int is_forced(int64_t i, int64_t n, int n_sink, int n_local)
{
    return i < n_sink || i >= n - n_local;
}

/* scores outside [2^-38, 1] (or NaN) are clamped into it */
static float tau_eff(float t)
{
    return t > VKO_TAU_FLOOR ? (t < 1.0f ? t : 1.0f) : VKO_TAU_FLOOR;
}

double vko_u128_to_double(uint64_t hi, uint64_t lo)
{
    unsigned __int128 v = ((unsigned __int128)hi << 64) | lo;
    return (double)v;
}

int vko_waterfill(int64_t n, const float* tau_in, int n_sink, int n_local, double budget,
                  double* c_out, int64_t* t_out, double* r64, float* r32)
{
    float* tau = (float*)malloc(sizeof(float) * (size_t)(n + 1));
    for (int64_t i = 0; i < n; ++i) tau[i] = tau_eff(tau_in[i]);
    int64_t n_forced = 0;
    for (int64_t i = 0; i < n; ++i) n_forced += is_forced(i, n, n_sink, n_local);
    const double bprime = budget - (double)n_forced;
    const int64_t n_u = n - n_forced;
    if (!(bprime > 0.0)) { free(tau); return -1; }
    double c;
    int64_t tstar = 0;
    if (bprime >= (double)n_u) {
        c = INFINITY;
        tstar = n_u;
    } else {
        int64_t* ord = (int64_t*)malloc(sizeof(int64_t) * (size_t)n_u);
        int64_t k = 0;
        for (int64_t i = 0; i < n; ++i) if (!is_forced(i, n, n_sink, n_local)) ord[k++] = i;
        g_sort_tau = tau;
        qsort(ord, (size_t)n_u, sizeof(int64_t), cmp_tau_desc);
        /* suffix sums in fixed point: tau * 2^61 is an integer for tau >= 2^-38 */
        unsigned __int128* suf = (unsigned __int128*)malloc(sizeof(unsigned __int128) * (size_t)(n_u + 1));
        suf[n_u] = 0;
        for (int64_t j = n_u - 1; j >= 0; --j) {
            double fx = ldexp((double)tau[ord[j]], 61);
            suf[j] = suf[j + 1] + (unsigned __int128)(uint64_t)fx;
        }
        double s = 0.0;
        for (tstar = 0; tstar < n_u; ++tstar) {
            s = ldexp((double)suf[tstar], -61);
            double lhs = (bprime - (double)tstar) * (double)tau[ord[tstar]];
            if (lhs < s) break;
        }
        c = (bprime - (double)tstar) / s;
        free(suf);
        free(ord);
    }
    for (int64_t i = 0; i < n; ++i) {
        double r;
        if (is_forced(i, n, n_sink, n_local)) r = 1.0;
        else {
            double ct = c * (double)tau[i];
            r = ct < 1.0 ? ct : 1.0;
        }
        if (r64) r64[i] = r;
        if (r32) r32[i] = (float)r;
    }
    *c_out = c;
    if (t_out) *t_out = tstar;
    free(tau);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* H/L split and Poisson sample (Algorithm 1, split and sampling steps).     */
/* ------------------------------------------------------------------------ */
void vko_poisson_sample(int64_t n, const float* r32, uint64_t seed, uint32_t kv_head,
                        uint32_t layer, uint32_t seq, uint8_t* flags)
{
    for (int64_t i = 0; i < n; ++i) {
        if (r32[i] == 1.0f) { flags[i] = 2; continue; }
        float u = vko_uniform(seed, (uint32_t)i, kv_head, layer, seq);
        flags[i] = (u < r32[i]) ? 1 : 0;
    }
}

/* ------------------------------------------------------------------------ */
/* Key sketches (Appendix A.1 and the int8 alternative).                     */
/* int8: per token s = max_c |k_c| / 127 in fp32, code = rint(k_c / s)       */
/*       clamped to [-127, 127]; s == 0 gives all-zero codes.                */
/* 2-bit: the d/8 rotate-half channel pairs (p, p + d/2) with the largest    */
/*       mean key energy; each kept channel quantised to 2 bits between the  */
/*       minimum and maximum of each group of `group` consecutive tokens,    */
/*       with an fp16 zero point (= min) and fp16 scale (= (max - min) / 3).  */
/* All code arithmetic is IEEE fp32 (codes are data and must match exactly). */
/* ------------------------------------------------------------------------ */
void vko_sketch_int8(int64_t n, int d, const float* K, int8_t* codes, float* scale)
{
    for (int64_t i = 0; i < n; ++i) {
        float mx = 0.0f;
        for (int c = 0; c < d; ++c) {
            float a = fabsf(K[(size_t)i * d + c]);
            if (a > mx) mx = a;
        }
        float s = mx / 127.0f;
        scale[i] = s;
        for (int c = 0; c < d; ++c) {
            int q = 0;
            if (s > 0.0f) {
                float v = rintf(K[(size_t)i * d + c] / s);
                if (v > 127.0f) v = 127.0f;
                if (v < -127.0f) v = -127.0f;
                q = (int)v;
            }
            codes[(size_t)i * d + c] = (int8_t)q;
        }
    }
}

static uint16_t f32_to_f16_bits(float x)
{
    _Float16 h = (_Float16)x;
    uint16_t b;
    memcpy(&b, &h, 2);
    return b;
}

static float f16_bits_to_f32(uint16_t b)
{
    _Float16 h;
    memcpy(&h, &b, 2);
    return (float)h;
}

float vko_f16_to_f32(uint16_t b) { return f16_bits_to_f32(b); }

/* pairs_out: d/8 pair indices p in [0, d/2), ascending.  Kept channel j is
 * pairs[j] for j < d/8 and pairs[j - d/8] + d/2 otherwise.
 * codes: [n][d/4] one code (0..3) per byte; zero/scale: [ngroups][d/4]. */
void vko_sketch_2bit(int64_t n, int d, const float* K, int group, int32_t* pairs_out,
                     uint8_t* codes, uint16_t* zero_h, uint16_t* scale_h)
{
    const int half = d / 2, npairs = d / 8, kept = d / 4;
    double* energy = (double*)calloc((size_t)half, sizeof(double));
    for (int64_t i = 0; i < n; ++i)
        for (int p = 0; p < half; ++p) {
            double a = K[(size_t)i * d + p], b = K[(size_t)i * d + p + half];
            energy[p] += a * a + b * b;
        }
    char* taken = (char*)calloc((size_t)half, 1);
    for (int j = 0; j < npairs; ++j) {
        int best = -1;
        for (int p = 0; p < half; ++p)
            if (!taken[p] && (best < 0 || energy[p] > energy[best])) best = p;
        taken[best] = 1;
    }
    int j = 0;
    for (int p = 0; p < half; ++p) if (taken[p]) pairs_out[j++] = p;
    int* ch = (int*)malloc(sizeof(int) * (size_t)kept);
    for (int q = 0; q < npairs; ++q) { ch[q] = pairs_out[q]; ch[q + npairs] = pairs_out[q] + half; }
    const int64_t ngroups = (n + group - 1) / group;
    for (int64_t g = 0; g < ngroups; ++g) {
        int64_t i0 = g * group, i1 = i0 + group < n ? i0 + group : n;
        for (int q = 0; q < kept; ++q) {
            float mn = INFINITY, mx = -INFINITY;
            for (int64_t i = i0; i < i1; ++i) {
                float v = K[(size_t)i * d + ch[q]];
                if (v < mn) mn = v;
                if (v > mx) mx = v;
            }
            uint16_t zb = f32_to_f16_bits(mn);
            uint16_t sb = f32_to_f16_bits((mx - mn) / 3.0f);
            zero_h[(size_t)g * kept + q] = zb;
            scale_h[(size_t)g * kept + q] = sb;
            float zf = f16_bits_to_f32(zb), sf = f16_bits_to_f32(sb);
            for (int64_t i = i0; i < i1; ++i) {
                int code = 0;
                if (sf > 0.0f) {
                    float v = rintf((K[(size_t)i * d + ch[q]] - zf) / sf);
                    if (v < 0.0f) v = 0.0f;
                    if (v > 3.0f) v = 3.0f;
                    code = (int)v;
                }
                codes[(size_t)i * kept + q] = (uint8_t)code;
            }
        }
    }
    free(ch);
    free(taken);
    free(energy);
}

/* ------------------------------------------------------------------------ */
/* Logits <q, k_i>/sqrt(d) in double: exact keys, and the sketch estimates   */
/* k^_i (int8: s_i * code_i; 2-bit: zero + scale * code on kept channels,    */
/* dropped channels contribute nothing).                                     */
/* ------------------------------------------------------------------------ */
void vko_logits_exact(int64_t n, int d, const double* q, const double* K, double* out)
{
    const double sd = sqrt((double)d);
    for (int64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += q[c] * K[(size_t)i * d + c];
        out[i] = s / sd;
    }
}

void vko_logits_int8(int64_t n, int d, const double* q, const int8_t* codes, const float* scale, double* out)
{
    const double sd = sqrt((double)d);
    for (int64_t i = 0; i < n; ++i) {
        double s = 0.0;
        for (int c = 0; c < d; ++c) s += q[c] * ((double)scale[i] * (double)codes[(size_t)i * d + c]);
        out[i] = s / sd;
    }
}

void vko_logits_2bit(int64_t n, int d, const double* q, const int32_t* pairs, const uint8_t* codes,
                     const uint16_t* zero_h, const uint16_t* scale_h, int group, double* out)
{
    const double sd = sqrt((double)d);
    const int half = d / 2, npairs = d / 8, kept = d / 4;
    for (int64_t i = 0; i < n; ++i) {
        const int64_t g = i / group;
        double s = 0.0;
        for (int qn = 0; qn < kept; ++qn) {
            int ch = qn < npairs ? pairs[qn] : pairs[qn - npairs] + half;
            double z = f16_bits_to_f32(zero_h[(size_t)g * kept + qn]);
            double sc = f16_bits_to_f32(scale_h[(size_t)g * kept + qn]);
            double khat = z + sc * (double)codes[(size_t)i * kept + qn];
            s += q[ch] * khat;
        }
        out[i] = s / sd;
    }
}

/* ------------------------------------------------------------------------ */
/* Bounded shrinkage estimator (Definition 2, eq. (5)) for one query row.    */
/* Inputs over L: w (sketch weights w^_i), r.                                */
/* lambda_i(beta) = clip_[r_i,1](beta r_i / (w_i (1 - r_i))) and beta is the */
/* fixed point beta = sum_L w_i (1 - lambda_i(beta)).  Exact breakpoint      */
/* enumeration: G(beta) = beta - sum_L w_i (1 - lambda_i(beta)) is           */
/* increasing and piecewise linear with breakpoints a_i = w_i (1 - r_i)     */
/* (below: lambda = r) and a_i / r_i (above: lambda = 1).  Sort the          */
/* breakpoints, find the segment where G changes sign by bisection over the  */
/* sorted list (G evaluated by a full sum each time), and solve the linear   */
/* equation on that segment.                                                 */
/* ------------------------------------------------------------------------ */
static double lambda_of(double beta, double w, double r)
{
    if (!(w > 0.0)) return 1.0;
    double x = beta * r / (w * (1.0 - r));
    if (x < r) x = r;
    if (x > 1.0) x = 1.0;
    return x;
}

static double G_of(double beta, int64_t nl, const double* w, const double* r)
{
    double f = 0.0;
    for (int64_t j = 0; j < nl; ++j) f += w[j] * (1.0 - lambda_of(beta, w[j], r[j]));
    return beta - f;
}

static int cmp_double(const void* a, const void* b)
{
    double x = *(const double*)a, y = *(const double*)b;
    return (x > y) - (x < y);
}

double vko_beta_breakpoints(int64_t nl, const double* w, const double* r)
{
    if (nl == 0) return 0.0;
    int64_t nb = 2 * nl + 1;
    double* bp = (double*)malloc(sizeof(double) * (size_t)nb);
    bp[0] = 0.0;
    for (int64_t j = 0; j < nl; ++j) {
        bp[1 + 2 * j] = w[j] * (1.0 - r[j]);
        bp[2 + 2 * j] = w[j] * (1.0 - r[j]) / r[j];
    }
    qsort(bp, (size_t)nb, sizeof(double), cmp_double);
    /* smallest k with G(bp[k]) >= 0; G(bp[nb-1]) = bp[nb-1] >= 0 */
    int64_t lo = 0, hi = nb - 1;
    if (G_of(bp[0], nl, w, r) >= 0.0) { double b0 = bp[0]; free(bp); return b0; }
    while (hi - lo > 1) {
        int64_t mid = lo + (hi - lo) / 2;
        if (G_of(bp[mid], nl, w, r) >= 0.0) hi = mid; else lo = mid;
    }
    double left = bp[lo], right = bp[hi];
    double beta;
    if (G_of(right, nl, w, r) == 0.0 || right == left) {
        beta = right;
    } else {
        /* on (left, right) every lambda_i is either constant or linear in beta */
        double mid = 0.5 * (left + right);
        double A = 0.0, W = 0.0, R = 0.0;
        for (int64_t j = 0; j < nl; ++j) {
            double aj = w[j] * (1.0 - r[j]);
            double gj = aj / r[j];
            if (!(w[j] > 0.0)) continue;
            if (mid <= aj) A += aj;                    /* lambda = r_j */
            else if (mid >= gj) { }                    /* lambda = 1 */
            else { W += w[j]; R += r[j] / (1.0 - r[j]); } /* interior */
        }
        beta = (A + W) / (1.0 + R);
    }
    free(bp);
    return beta;
}

/* ------------------------------------------------------------------------ */
/* Binary shrinkage ("Verify Before You Fetch", App. A.2): every lambda_i is */
/* one of the endpoints {1, r_i}.  Turning token i from 1 to r_i changes the */
/* MSE of eq. (6) by w_i (1 - r_i) (2 beta - w_i (1 - r_i) / r_i), beta being */
/* the bias already accumulated, so the tokens of L are visited by          */
/* decreasing gamma_i = w_i (1 - r_i) / r_i (ties: lower L index first) and  */
/* set to r_i while gamma_i > 2 beta; the others keep lambda = 1.  Writes    */
/* lambda (length nl) and returns the final beta = sum of w_i (1 - r_i) over */
/* the tokens set to r_i.                                                    */
/* ------------------------------------------------------------------------ */
static _Thread_local const double* g_sort_gam;
static int cmp_gamma_desc(const void* a, const void* b)
{
    int64_t ia = *(const int64_t*)a, ib = *(const int64_t*)b;
    double ga = g_sort_gam[ia], gb = g_sort_gam[ib];
    if (ga > gb) return -1;
    if (ga < gb) return 1;
    return (ia < ib) ? -1 : (ia > ib);
}

double vko_binary_shrinkage(int64_t nl, const double* w, const double* r, double* lam, int64_t* n_shrunk)
{
    double* gam = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
    int64_t* ord = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nl + 1));
    for (int64_t j = 0; j < nl; ++j) {
        gam[j] = w[j] * (1.0 - r[j]) / r[j];
        ord[j] = j;
        lam[j] = 1.0;
    }
    g_sort_gam = gam;
    qsort(ord, (size_t)nl, sizeof(int64_t), cmp_gamma_desc);
    double beta = 0.0;
    int64_t k = 0;
    for (; k < nl; ++k) {
        int64_t j = ord[k];
        if (!(gam[j] > 2.0 * beta)) break;
        lam[j] = r[j];
        beta += w[j] * (1.0 - r[j]);
    }
    if (n_shrunk) *n_shrunk = k;
    free(gam);
    free(ord);
    return beta;
}

/* ------------------------------------------------------------------------ */
/* Bernstein certificate (Lemma 1, eq. (7)) over a subset of L, with fixed  */
/* per-token coefficients.  a_i = w_i (1 - lambda_i), v_i = lambda_i^2 w_i^2 */
/* (1 - r_i) / r_i, b_i = lambda_i w_i / r_i * max(r_i, 1 - r_i).  Empty     */
/* sums and maxima are zero.                                                 */
/* ------------------------------------------------------------------------ */
static double cert_from_sums(double sa, double sv, double bmax, double ldelta, double D)
{
    double t = bmax * ldelta / 3.0;
    return (sa + t + sqrt(t * t + 2.0 * sv * ldelta)) / D;
}

typedef struct {
    double m;        /* logit shift */
    double D;        /* certificate denominator: sum_H w_i + sum_L w^_i */
    double beta;     /* fixed point of Definition 2 */
    double sum_a;    /* beta(L) of eq. (7) */
    double V;        /* V(L) */
    double b;        /* b(L) */
    double eps_hat;  /* eq. (7) on the whole of L */
    int64_t n_l;
    int64_t kstar;
    int32_t no_fetch;
    int32_t pad;
} vko_cert;

static _Thread_local const double* g_sort_g;
static _Thread_local const int64_t* g_sort_idx;
static int cmp_gain(const void* a, const void* b)
{
    int64_t ia = *(const int64_t*)a, ib = *(const int64_t*)b;
    double ga = g_sort_g[ia], gb = g_sort_g[ib];
    if (ga > gb) return -1;
    if (ga < gb) return 1;
    int64_t ta = g_sort_idx[ia], tb = g_sort_idx[ib];
    return (ta < tb) ? -1 : (ta > tb);
}

/*
 * KVFetch for one query row (Algorithm 2).
 *   flags[n], r32[n]      : compressed state of the row's KV head.
 *   t_exact[n]            : exact logits (used on H).
 *   t_sketch[n]           : sketch logits (used on all of L).
 *   eps, delta            : tolerance.
 *   mode                  : 0 = definition (every eps^(L\{i}) and every
 *                           eps^(L_g[k:]) recomputed from scratch, O(|L|^2));
 *                           1 = algebraically identical closed forms
 *                           (leave-one-out sums, tail sums), O(|L| log |L|).
 * Outputs (any pointer may be NULL):
 *   cert                  : scalars.
 *   lambda[n]             : lambda_i on L (0 elsewhere).
 *   gain[n]               : g_i on L when the row fetches (0 elsewhere).
 *   order[|L|]            : L sorted by gain descending, ties by token index.
 *   exact_mask[n]         : 1 for the tokens of L_g[:k*] (made exact).
 *   resid[|L| + 1]        : eps^(L_g[k:]) for k = 0..|L| (from tail sums; for diagnostics).
 * Returns 0.
 */
int vko_kvfetch_row_ex(int64_t n, const uint8_t* flags, const float* r32, const double* t_exact,
                       const double* t_sketch, const uint8_t* use_exact, double eps, double delta, int mode,
                       int shrinkage, vko_cert* cert, double* lambda, double* gain, int64_t* order,
                       uint8_t* exact_mask, double* resid);

int vko_kvfetch_row(int64_t n, const uint8_t* flags, const float* r32, const double* t_exact,
                    const double* t_sketch, double eps, double delta, int mode, vko_cert* cert,
                    double* lambda, double* gain, int64_t* order, uint8_t* exact_mask, double* resid)
{
    return vko_kvfetch_row_ex(n, flags, r32, t_exact, t_sketch, NULL, eps, delta, mode, 0, cert, lambda, gain,
                              order, exact_mask, resid);
}

/* shrinkage: 0 = the clipped coefficients of Definition 2, 1 = binary (App. A.2).
 * use_exact[n] (or NULL): tokens of L whose exact logit replaces the sketch logit in every quantity of
 * the decision (App. A.1: resident and shortlisted tokens). */
int vko_kvfetch_row_ex(int64_t n, const uint8_t* flags, const float* r32, const double* t_exact,
                       const double* t_sketch, const uint8_t* use_exact, double eps, double delta, int mode,
                       int shrinkage, vko_cert* cert, double* lambda, double* gain, int64_t* order,
                       uint8_t* exact_mask, double* resid)
{
    int64_t nl = 0;
    double m = -INFINITY;
#define VKO_T_OF(i) ((use_exact && use_exact[i]) ? t_exact[i] : t_sketch[i])
    for (int64_t i = 0; i < n; ++i) {
        if (flags[i] == 2) { if (t_exact[i] > m) m = t_exact[i]; }
        else { ++nl; if (VKO_T_OF(i) > m) m = VKO_T_OF(i); }
    }
    int64_t* lidx = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nl + 1));
    double* w = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
    double* r = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
    double D = 0.0;
    int64_t k = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (flags[i] == 2) D += exp(t_exact[i] - m);
        else {
            lidx[k] = i;
            w[k] = exp(VKO_T_OF(i) - m);
            r[k] = (double)r32[i];
            D += w[k];
            ++k;
        }
    }
    const double ldelta = log(2.0 / delta);
    double* lamb = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
    double beta;
    if (shrinkage == 1) {
        beta = vko_binary_shrinkage(nl, w, r, lamb, NULL);
    } else {
        beta = vko_beta_breakpoints(nl, w, r);
        for (int64_t j = 0; j < nl; ++j) lamb[j] = lambda_of(beta, w[j], r[j]);
    }
    double* a = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
    double* v = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
    double* bb = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
    double sa = 0.0, sv = 0.0, bmax = 0.0;
    if (lambda) for (int64_t i = 0; i < n; ++i) lambda[i] = 0.0;
    for (int64_t j = 0; j < nl; ++j) {
        double lam = lamb[j];
        if (lambda) lambda[lidx[j]] = lam;
        a[j] = w[j] * (1.0 - lam);
        v[j] = lam * lam * w[j] * w[j] * (1.0 - r[j]) / r[j];
        double mr = r[j] > 1.0 - r[j] ? r[j] : 1.0 - r[j];
        bb[j] = lam * w[j] / r[j] * mr;
        sa += a[j];
        sv += v[j];
        if (bb[j] > bmax) bmax = bb[j];
    }
    double eh = cert_from_sums(sa, sv, bmax, ldelta, D);
    int no_fetch = eh < eps;
    int64_t kstar = 0;
    if (gain) for (int64_t i = 0; i < n; ++i) gain[i] = 0.0;
    if (exact_mask) for (int64_t i = 0; i < n; ++i) exact_mask[i] = 0;
    int64_t* ord = (int64_t*)malloc(sizeof(int64_t) * (size_t)(nl + 1));
    for (int64_t j = 0; j < nl; ++j) ord[j] = j;
    if (!no_fetch) {
        double* g = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
        if (mode == 0) {
            /* eq. (9) as written: g_i = eps^(L) - eps^(L \ {i}) */
            for (int64_t i = 0; i < nl; ++i) {
                double s1 = 0.0, s2 = 0.0, b1 = 0.0;
                for (int64_t j = 0; j < nl; ++j) {
                    if (j == i) continue;
                    s1 += a[j];
                    s2 += v[j];
                    if (bb[j] > b1) b1 = bb[j];
                }
                g[i] = eh - cert_from_sums(s1, s2, b1, ldelta, D);
            }
        } else {
            /* the same difference written without cancellation:
             * g_i = [a_i + (b - b_-i) l/3 + (A - A_-i) / (sqrt(A) + sqrt(A_-i))] / D,
             * A = (b l/3)^2 + 2 V l, A_-i = (b_-i l/3)^2 + 2 (V - v_i) l */
            double b1 = -1.0, b2 = 0.0;
            int64_t arg = -1;
            for (int64_t j = 0; j < nl; ++j) {
                if (bb[j] > b1) { b2 = b1 < 0 ? 0.0 : b1; b1 = bb[j]; arg = j; }
                else if (bb[j] > b2) b2 = bb[j];
            }
            if (b1 < 0) b1 = 0.0;
            const double t = b1 * ldelta / 3.0;
            const double A = t * t + 2.0 * sv * ldelta;
            for (int64_t i = 0; i < nl; ++i) {
                double bmi = (i == arg) ? b2 : b1;
                double tm = bmi * ldelta / 3.0;
                double vmi = sv - v[i];
                if (vmi < 0.0) vmi = 0.0;
                double Ami = tm * tm + 2.0 * vmi * ldelta;
                double dA = (t * t - tm * tm) + 2.0 * v[i] * ldelta;
                double den = sqrt(A) + sqrt(Ami);
                double root = den > 0.0 ? dA / den : 0.0;
                g[i] = (a[i] + (t - tm) + root) / D;
            }
        }
        g_sort_g = g;
        g_sort_idx = lidx;
        qsort(ord, (size_t)nl, sizeof(int64_t), cmp_gain);
        /* eq. (10): smallest k with eps^(L_g[k:]) < eps; k = |L| always accepted */
        if (mode == 0) {
            for (kstar = 0; kstar < nl; ++kstar) {
                double s1 = 0.0, s2 = 0.0, b1 = 0.0;
                for (int64_t p = kstar; p < nl; ++p) {
                    int64_t j = ord[p];
                    s1 += a[j];
                    s2 += v[j];
                    if (bb[j] > b1) b1 = bb[j];
                }
                if (cert_from_sums(s1, s2, b1, ldelta, D) < eps) break;
            }
        } else {
            double* ts = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
            double* tv = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
            double* tb = (double*)malloc(sizeof(double) * (size_t)(nl + 1));
            ts[nl] = 0.0; tv[nl] = 0.0; tb[nl] = 0.0;
            for (int64_t p = nl - 1; p >= 0; --p) {
                int64_t j = ord[p];
                ts[p] = ts[p + 1] + a[j];
                tv[p] = tv[p + 1] + v[j];
                tb[p] = bb[j] > tb[p + 1] ? bb[j] : tb[p + 1];
            }
            for (kstar = 0; kstar < nl; ++kstar)
                if (cert_from_sums(ts[kstar], tv[kstar], tb[kstar], ldelta, D) < eps) break;
            free(ts); free(tv); free(tb);
        }
        if (resid) {
            double s1 = 0.0, s2 = 0.0, b1 = 0.0;
            resid[nl] = 0.0;
            for (int64_t p = nl - 1; p >= 0; --p) {
                int64_t j = ord[p];
                s1 += a[j];
                s2 += v[j];
                if (bb[j] > b1) b1 = bb[j];
                resid[p] = cert_from_sums(s1, s2, b1, ldelta, D);
            }
        }
        if (gain) for (int64_t j = 0; j < nl; ++j) gain[lidx[j]] = g[j];
        if (exact_mask) for (int64_t p = 0; p < kstar; ++p) exact_mask[lidx[ord[p]]] = 1;
        free(g);
    }
    if (order) for (int64_t p = 0; p < nl; ++p) order[p] = lidx[ord[p]];
    if (cert) {
        cert->m = m; cert->D = D; cert->beta = beta; cert->sum_a = sa; cert->V = sv;
        cert->b = bmax; cert->eps_hat = eh; cert->n_l = nl; cert->kstar = kstar;
        cert->no_fetch = no_fetch; cert->pad = 0;
    }
    free(ord); free(a); free(v); free(bb); free(lidx); free(w); free(r); free(lamb);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* The estimator of Definition 2 / eq. (5) after the fetch (Theorem 2):     */
/*   D^ = sum_H w_i + sum_{L_g[:k*]} w_i + sum_{S \ L_g[:k*]} lambda_i w_i / r_i */
/* and the numerator N^ with the same weights on the value rows, where w_i  */
/* = exp(t_i - m) is the EXACT weight (the keys of the sample are resident, */
/* those of L_g[:k*] are fetched).  Tokens of L outside the sample and not  */
/* fetched contribute nothing (their Z_i = 0).  flags encode the sample     */
/* outcome (1 = Z_i = 1).  Writes num[d] and returns D^ (units exp(-m)).     */
/* ------------------------------------------------------------------------ */
double vko_estimate_row(int64_t n, int d, const uint8_t* flags, const float* r32, const double* t_exact,
                        const double* V, const double* lambda, const uint8_t* exact_mask, double m, double* num)
{
    double den = 0.0;
    if (num) for (int c = 0; c < d; ++c) num[c] = 0.0;
    for (int64_t i = 0; i < n; ++i) {
        double om;
        if (flags[i] == 2 || (exact_mask && exact_mask[i])) om = 1.0;
        else if (flags[i] == 1) om = lambda[i] / (double)r32[i];
        else continue;
        double wt = om * exp(t_exact[i] - m);
        den += wt;
        if (num) for (int c = 0; c < d; ++c) num[c] += wt * V[(size_t)i * d + c];
    }
    return den;
}

/* ------------------------------------------------------------------------ */
/* Final attention (comment after Algorithm 2): o = N^ / D^ of the estimator */
/* above, the shift m taken as the largest logit of a token with nonzero     */
/* weight (any m gives the same ratio).                                      */
/* ------------------------------------------------------------------------ */
void vko_attention_row(int64_t n, int d, const uint8_t* flags, const float* r32, const double* t_exact,
                       const double* V, const double* lambda, const uint8_t* exact_mask, double* out)
{
    double m = -INFINITY;
    for (int64_t i = 0; i < n; ++i) {
        int live = flags[i] == 2 || flags[i] == 1 || (exact_mask && exact_mask[i]);
        if (live && t_exact[i] > m) m = t_exact[i];
    }
    double den = vko_estimate_row(n, d, flags, r32, t_exact, V, lambda, exact_mask, m, out);
    for (int c = 0; c < d; ++c) out[c] /= den;
}

/* ------------------------------------------------------------------------ */
/* Batched driver for the CPU baseline: independent rows in parallel.       */
/* Row u uses flags/r32 of kv row kv_of[u] and logits rows u.                */
/* ------------------------------------------------------------------------ */
/* ------------------------------------------------------------------------ */
/* Shortlist ("Verify Before You Fetch", App. A.1): among the non-resident  */
/* tokens of L (flags 0) of one KV head, the k with the largest sketch      */
/* score over the head's G query rows (score = the largest sketch logit of  */
/* the token over the rows; ties: lower token index).  t_sketch is [G][n].  */
/* Sets mask[i] = 1 for them (mask is not cleared); returns how many.       */
/* ------------------------------------------------------------------------ */
static _Thread_local const double* g_sort_score;
static int cmp_score_desc(const void* a, const void* b)
{
    int64_t ia = *(const int64_t*)a, ib = *(const int64_t*)b;
    double sa = g_sort_score[ia], sb = g_sort_score[ib];
    if (sa > sb) return -1;
    if (sa < sb) return 1;
    return (ia < ib) ? -1 : (ia > ib);
}

int64_t vko_shortlist(int64_t n, int G, const uint8_t* flags, const double* t_sketch, int64_t k, uint8_t* mask)
{
    double* score = (double*)malloc(sizeof(double) * (size_t)(n + 1));
    int64_t* cand = (int64_t*)malloc(sizeof(int64_t) * (size_t)(n + 1));
    int64_t nc = 0;
    for (int64_t i = 0; i < n; ++i) {
        double sc = -INFINITY;
        for (int g = 0; g < G; ++g)
            if (t_sketch[(int64_t)g * n + i] > sc) sc = t_sketch[(int64_t)g * n + i];
        score[i] = sc;
        if (flags[i] == 0) cand[nc++] = i;
    }
    g_sort_score = score;
    qsort(cand, (size_t)nc, sizeof(int64_t), cmp_score_desc);
    const int64_t take = k < nc ? k : nc;
    for (int64_t j = 0; j < take; ++j) mask[cand[j]] = 1;
    free(score);
    free(cand);
    return take;
}

int vko_kvfetch_rows(int64_t rows, int64_t n, const uint8_t* flags, const float* r32, const int32_t* kv_of,
                     const double* t_exact, const double* t_sketch, double eps, double delta, int mode,
                     int shrinkage, vko_cert* certs, uint8_t* exact_masks, int threads)
{
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int64_t u = 0; u < rows; ++u) {
        const int64_t kv = kv_of[u];
        vko_kvfetch_row_ex(n, flags + kv * n, r32 + kv * n, t_exact + u * n, t_sketch + u * n, NULL, eps, delta,
                           mode, shrinkage, certs + u, NULL, NULL, NULL, exact_masks ? exact_masks + u * n : NULL,
                           NULL);
    }
    return 0;
}

int vko_num_threads(void)
{
#ifdef _OPENMP
    int t = 0;
#pragma omp parallel
    {
#pragma omp single
        t = omp_get_num_threads();
    }
    return t;
#else
    return 1;
#endif
}
